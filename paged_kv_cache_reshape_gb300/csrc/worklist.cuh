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
#pragma once
#include "step.h"
#include "../../include/pa.h"

namespace pa {
namespace worklist {

constexpr int kThreads = 1024;  // the builder runs in one CTA of this size

struct Int3 {
  int a, b, c, d, e;  // full decode splits, prefill tiles, combine rows, decode entries (last splits),
                      // split decode entries
};

// Exclusive scan of the five counters across the block (out of line: one
// copy of its code serves every call, which keeps the cold instruction
// fetches of the builder few); returns the prefix and
// writes the block totals to *tot.  All threads must call it.
__device__ __noinline__ Int3 block_exclusive_scan3(Int3 v, Int3* tot) {
  __shared__ Int3 warp_sums[32];
  __shared__ Int3 total;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  Int3 inc = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    int a = __shfl_up_sync(0xffffffffu, inc.a, o);
    int b = __shfl_up_sync(0xffffffffu, inc.b, o);
    int c = __shfl_up_sync(0xffffffffu, inc.c, o);
    int d = __shfl_up_sync(0xffffffffu, inc.d, o);
    int e = __shfl_up_sync(0xffffffffu, inc.e, o);
    if (lane >= o) {
      inc.a += a;
      inc.b += b;
      inc.c += c;
      inc.d += d;
      inc.e += e;
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
      int d = __shfl_up_sync(0xffffffffu, wi.d, o);
      int e = __shfl_up_sync(0xffffffffu, wi.e, o);
      if (lane >= o) {
        wi.a += a;
        wi.b += b;
        wi.c += c;
        wi.d += d;
        wi.e += e;
      }
    }
    warp_sums[lane] = Int3{wi.a - w.a, wi.b - w.b, wi.c - w.c, wi.d - w.d, wi.e - w.e};
    if (lane == 31) total = wi;
  }
  __syncthreads();
  *tot = total;
  Int3 base = warp_sums[warp];
  Int3 out{base.a + inc.a - v.a, base.b + inc.b - v.b, base.c + inc.c - v.c, base.d + inc.d - v.d,
           base.e + inc.e - v.e};
  __syncthreads();
  return out;
}

__device__ __noinline__ long long block_sum_ll(long long v) {
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

__device__ int route_of(const WorklistParams& p, int q) {
  const long long rows = (long long)q * p.group;
  if (rows <= p.dec_max_rows) return kRouteDecode;
  if (p.chunk_tokens > 0 && (p.chunk_rows_max <= 0 || rows <= p.chunk_rows_max)) return kRouteChunked;
  return kRoutePrefill;
}

// First key position a row at `past` (the earliest new token) may attend,
// aligned down to a 64-key stage: with a window W the earliest admitted
// position is past + 1 - W (section 9.2 block-table pruning).
__device__ int walk_start(const WorklistParams& p, int past) {
  int lo = 0;
  if (p.prune && p.window >= 1) lo = max(0, past + 1 - p.window);
  return lo & ~(kStageKeys - 1);
}

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
  L.lo = walk_start(p, past);
  L.route = route_of(p, q);
  return L;
}

// Decode-table entries of a sequence: the sequence itself (decode route)
// or its chunks of chunk_tokens tokens (chunked route).
struct Entry {
  int q, past, t0, lo;
};

__device__ int entry_count(const WorklistParams& p, const Lens& L) {
  if (L.route == kRouteDecode) return 1;
  if (L.route == kRouteChunked) return (L.q + p.chunk_tokens - 1) / p.chunk_tokens;
  return 0;
}

__device__ Entry entry_of(const WorklistParams& p, const Lens& L, int c) {
  if (L.route == kRouteDecode) return Entry{L.q, L.past, L.t0, L.lo};
  const int ct = p.chunk_tokens;
  Entry e;
  e.q = min(ct, L.q - c * ct);
  e.past = L.past + c * ct;
  e.t0 = L.t0 + c * ct;
  e.lo = walk_start(p, e.past);
  return e;
}

// Keys an entry walks, and its splits.
__device__ int entry_span(const Entry& e) { return e.past + e.q - e.lo; }
__device__ int entry_splits(const Entry& e, int split_keys) { return (entry_span(e) + split_keys - 1) / split_keys; }

// Decode keys a sequence's entries walk (they set the split size).
__device__ long long decode_span(const WorklistParams& p, const Lens& L) {
  long long span = 0;
  const int n = entry_count(p, L);
  for (int c = 0; c < n; ++c) span += entry_span(entry_of(p, L, c));
  return span;
}

// Counts of one sequence: a = full decode splits, b = prefill tiles, c =
// combine rows, d = decode entries (one last split each), e = split
// entries (a + e split-partial slots).
__device__ Int3 seq_counts(const WorklistParams& p, const Lens& L, int split_keys) {
  Int3 cnt{0, 0, 0, 0, 0};
  const int n = entry_count(p, L);
  for (int c = 0; c < n; ++c) {
    const Entry e = entry_of(p, L, c);
    const int ns = entry_splits(e, split_keys);
    cnt.a += ns - 1;
    if (ns > 1) {
      cnt.c += e.q;
      cnt.e += 1;
    }
  }
  cnt.d = n;
  if (L.route == kRoutePrefill) cnt.b = (L.q + p.prefill_tile_tokens - 1) / p.prefill_tile_tokens;
  return cnt;
}

// Writes the decode-table entries of sequence b (the first at index v0),
// their full splits from item a0 on, their combine rows from row c0 on and
// their split-partial slots from slot s0 on; last_item(c, entry, splits)
// gives the item index of entry c's last split.
template <typename LastItem>
__device__ void write_entries(const WorklistParams& p, const Lens& L, int b, int v0, int a0, int c0, int s0,
                              int split_keys, LastItem last_item) {
  const int n = entry_count(p, L);
  for (int c = 0; c < n; ++c) {
    const Entry e = entry_of(p, L, c);
    const int ns = entry_splits(e, split_keys);
    const int v = v0 + c;
    SeqInfo d;
    d.q_len = e.q;
    d.kv_len = e.past + e.q;
    d.lo = e.lo;
    d.t0 = e.t0;
    d.dec_first = a0;
    d.dec_count = ns;
    d.dec_last = last_item(c, e, ns);
    d.pre_first = 0;
    d.pre_count = 0;
    d.comb_first = c0;
    d.b = b;
    d.part_first = ns > 1 ? s0 : -1;
    p.dseq[v] = d;
    for (int s = 0; s + 1 < ns; ++s) p.dec_items[a0 + s] = make_int2(v, s);
    p.dec_items[d.dec_last] = make_int2(v, ns - 1);
    if (ns > 1)
      for (int j = 0; j < e.q; ++j) p.comb_rows[c0 + j] = make_int2(e.t0 + j, v);
    a0 += ns - 1;
    if (ns > 1) {
      c0 += e.q;
      s0 += ns;
    }
  }
}

// Sequence-table entry of sequence b.
__device__ void write_seq(const WorklistParams& p, const Lens& L, int b, int pre_first, int pre_count) {
  SeqInfo si;
  si.q_len = L.q;
  si.kv_len = L.past + L.q;
  si.lo = L.lo;
  si.t0 = L.t0;
  si.dec_first = si.dec_count = si.dec_last = 0;
  si.pre_first = pre_first;
  si.pre_count = pre_count;
  si.comb_first = 0;
  si.b = b;
  si.part_first = 0;
  p.seq[b] = si;
}

// (query token, admitted key) pairs of a prefill-routed sequence, for the
// SM split's cost model (the window's cut is ignored: an estimate).
__device__ long long prefill_pairs(const Lens& L) {
  return L.route == kRoutePrefill ? (long long)L.q * (L.past + (L.q + 1) / 2) : 0;
}

__device__ int split_keys_for(const WorklistParams& p, long long total) {
  if (p.split_keys_fixed > 0) return p.split_keys_fixed;
  long long per = (total + p.target_pairs - 1) / max(p.target_pairs, 1);
  per = (per + kStageKeys - 1) / kStageKeys * kStageKeys;
  return (int)min(max(per, (long long)max(p.min_split_keys, kStageKeys)), (long long)(1 << 30));
}

// SM split for a step with both decode and prefill work: the prefill CTAs
// kept, P, minimise max(prefill time on P SMs, decode time on the rest),
// with prefill time = FLOPs / (P * per-SM rate) and decode time = K/V bytes
// / min(HBM rate, SMs * per-SM rate).  Without one of the two kinds of
// work, or without a split, every launched CTA takes work.
__device__ void choose_split(const WorklistParams& p, long long dec_keys, long long pre_pairs, Counters* c) {
  c->pre_ctas = p.pre_grid;
  c->dec_ctas = p.dec_grid;
  if (p.split_sms < 2 || dec_keys <= 0 || pre_pairs <= 0) return;
  if (p.force_pre_ctas > 0) {  // a fixed share (a tuning and test option)
    c->pre_ctas = min(min(p.force_pre_ctas, p.split_sms - 1), p.pre_grid);
    c->dec_ctas = max(1, min(p.dec_grid, (p.split_sms - c->pre_ctas) * p.dec_ctas_per_sm));
    return;
  }
  const float F = (float)pre_pairs * p.pre_flops_per_pair;
  const float B = (float)dec_keys * p.dec_bytes_per_key;
  int best = 1;
  float best_t = 3.0e38f;
  for (int P = 1; P < p.split_sms; ++P) {
    const float t_pre = F / ((float)P * p.pre_rate_sm);
    const float t_dec = B / fminf(p.hbm_rate, (float)(p.split_sms - P) * p.dec_rate_sm);
    const float t = fmaxf(t_pre, t_dec);
    if (t < best_t) {
      best_t = t;
      best = P;
    }
  }
  c->pre_ctas = min(best, p.pre_grid);
  c->dec_ctas = max(1, min(p.dec_grid, (p.split_sms - c->pre_ctas) * p.dec_ctas_per_sm));
}

__device__ void write_counters(const WorklistParams& p, bool overflow, Int3 tot, int split_keys, long long dec_keys,
                               long long pre_pairs, int* err_bits) {
  Counters c;
  if (overflow) *err_bits |= PA_DEVERR_KV_BOUND;
  c.n_dec = overflow ? 0 : tot.a + tot.d;
  c.n_pre = overflow ? 0 : tot.b;
  c.n_comb = overflow ? 0 : tot.c;
  c.split_keys = split_keys;
  c.dec_next = 0;
  c.pre_next = 0;
  choose_split(p, dec_keys, pre_pairs, &c);
  c.pad[0] = c.pad[1] = c.pad[2] = c.pad[3] = 0;
  *p.counters = c;
}

// Batches of at most one CTA's width: every sequence stays in its thread's
// registers from the length read to the item writes (one pass).
__device__ void build_small(const WorklistParams& p) {
  int err_bits = 0;
  const int b = threadIdx.x;
  Lens L{0, 0, 0, 0, kRouteNone};
  if (b < p.batch) L = read_lens(p, b, &err_bits);
  const long long dec_keys = block_sum_ll(decode_span(p, L));
  // the prefill side of the SM split's cost model (no split: not needed)
  const long long pre_pairs = p.split_sms >= 2 ? block_sum_ll(prefill_pairs(L)) : 0;
  const int split_keys = split_keys_for(p, dec_keys);
  const Int3 cnt = seq_counts(p, L, split_keys);
  Int3 tot;
  const Int3 pre = block_exclusive_scan3(cnt, &tot);
  const bool overflow = tot.a + tot.d > p.cap_dec || tot.b > p.cap_pre || tot.c > p.cap_comb ||
                        tot.d > p.cap_dseq || tot.a + tot.e > p.cap_part;
  // Last splits, longest first: they are the only items shorter than
  // split_keys, so handing them out in decreasing size keeps the dynamic
  // queue's tail short.  Bucket = 64-key groups, counting sort; an entry's
  // place within its bucket comes from an atomic (the item order does not
  // change any result).
  __shared__ int hist[kThreads];
  hist[threadIdx.x] = 0;
  __syncthreads();
  const int n_e = cnt.d;
  auto last_bucket = [&](const Entry& e, int ns) {
    const int last = entry_span(e) - (ns - 1) * split_keys;  // keys of the last split, >= 1
    return kThreads - 1 - min(kThreads - 1, (last - 1) / kStageKeys);
  };
  for (int c = 0; c < n_e; ++c) {
    const Entry e = entry_of(p, L, c);
    atomicAdd(&hist[last_bucket(e, entry_splits(e, split_keys))], 1);
  }
  __syncthreads();
  Int3 htot;
  const Int3 hpre = block_exclusive_scan3(Int3{hist[threadIdx.x], 0, 0, 0, 0}, &htot);
  __syncthreads();
  hist[threadIdx.x] = hpre.a;
  __syncthreads();
  if (b < p.batch) {
    write_seq(p, L, b, pre.b, cnt.b);
    if (!overflow)
      write_entries(p, L, b, pre.d, pre.a, pre.c, pre.a + pre.e, split_keys, [&](int, const Entry& e, int ns) {
        return tot.a + atomicAdd(&hist[last_bucket(e, ns)], 1);
      });
  }
  // Prefill tiles, costliest first (cost ~ the tile's last position, in
  // 64-key buckets): the same counting sort over every tile of every
  // sequence (skipped by the whole block when no sequence has a tile).
  if (tot.b > 0) {
    __syncthreads();
    hist[threadIdx.x] = 0;
    __syncthreads();
    auto tile_bucket = [&](int s) {
      const int pos_end = L.past + min((s + 1) * p.prefill_tile_tokens, L.q);
      return kThreads - 1 - min(kThreads - 1, pos_end / kStageKeys);
    };
    for (int s = 0; s < cnt.b; ++s) atomicAdd(&hist[tile_bucket(s)], 1);
    __syncthreads();
    const Int3 ppre = block_exclusive_scan3(Int3{hist[threadIdx.x], 0, 0, 0, 0}, &htot);
    __syncthreads();
    hist[threadIdx.x] = ppre.a;
    __syncthreads();
    if (!overflow)
      for (int s = 0; s < cnt.b; ++s) p.pre_tiles[atomicAdd(&hist[tile_bucket(s)], 1)] = make_int2(b, s);
  }
  if (threadIdx.x == 0) write_counters(p, overflow, tot, split_keys, dec_keys, pre_pairs, &err_bits);
  if (err_bits) atomicOr(p.err, err_bits);
}

// Batches of more than one CTA's width (kept out of line: its code is not
// fetched on the small-batch path).
__device__ __noinline__ void build_large(const WorklistParams& p) {
  int err_bits = 0;
  // Pass 1: total decode span, which sets the keys per split.
  long long span = 0, pairs = 0;
  for (int base = 0; base < p.batch; base += kThreads) {
    int b = base + threadIdx.x;
    if (b < p.batch) {
      int dummy = 0;
      const Lens L = read_lens(p, b, &dummy);
      span += decode_span(p, L);
      pairs += prefill_pairs(L);
    }
  }
  const long long dec_keys = block_sum_ll(span);
  const long long pre_pairs = p.split_sms >= 2 ? block_sum_ll(pairs) : 0;
  const int split_keys = split_keys_for(p, dec_keys);

  // Pass 2: counts and scans.  The totals fix where every list starts; the
  // number of full decode splits (which precede every last split) is known
  // only at the end, so the items are written in pass 3.  Last splits stay
  // in entry order here.
  Int3 carry{0, 0, 0, 0, 0};
  for (int base = 0; base < p.batch; base += kThreads) {
    int b = base + threadIdx.x;
    Lens L{0, 0, 0, 0, kRouteNone};
    Int3 cnt{0, 0, 0, 0, 0};
    if (b < p.batch) {
      L = read_lens(p, b, &err_bits);
      cnt = seq_counts(p, L, split_keys);
    }
    Int3 tot;
    const Int3 pre = block_exclusive_scan3(cnt, &tot);
    if (b < p.batch) {
      write_seq(p, L, b, carry.b + pre.b, cnt.b);
      // the prefixes pass 3 needs, kept in this sequence's entry
      p.seq[b].dec_first = carry.a + pre.a;
      p.seq[b].dec_last = carry.d + pre.d;  // first decode entry (and last split, before the full splits)
      p.seq[b].comb_first = carry.c + pre.c;
      p.seq[b].part_first = carry.a + carry.e + pre.a + pre.e;
      p.seq[b].dec_count = cnt.d;
    }
    carry.a += tot.a;
    carry.b += tot.b;
    carry.c += tot.c;
    carry.d += tot.d;
    carry.e += tot.e;
  }
  const int n_full = carry.a;
  const bool overflow = carry.a + carry.d > p.cap_dec || carry.b > p.cap_pre || carry.c > p.cap_comb ||
                        carry.d > p.cap_dseq || carry.a + carry.e > p.cap_part;
  __syncthreads();
  // Pass 3: decode entries, items and tiles (skipped if a list would overflow).
  if (!overflow) {
    for (int b = threadIdx.x; b < p.batch; b += kThreads) {
      const SeqInfo si = p.seq[b];
      if (si.dec_count > 0) {
        Lens L;
        L.q = si.q_len;
        L.past = si.kv_len - si.q_len;
        L.t0 = si.t0;
        L.lo = si.lo;
        L.route = route_of(p, si.q_len);
        write_entries(p, L, b, si.dec_last, si.dec_first, si.comb_first, si.part_first, split_keys,
                      [&](int c, const Entry&, int) { return n_full + si.dec_last + c; });
      }
      for (int s = 0; s < si.pre_count; ++s) p.pre_tiles[si.pre_first + s] = make_int2(b, s);
    }
  }
  if (threadIdx.x == 0) write_counters(p, overflow, carry, split_keys, dec_keys, pre_pairs, &err_bits);
  if (err_bits) atomicOr(p.err, err_bits);
}

// Body of the builder; must be executed by all kThreads threads of one CTA.
__device__ void build(const WorklistParams& p) {
  if (p.batch <= kThreads) build_small(p);
  else build_large(p);
}

}  // namespace worklist
}  // namespace pa
