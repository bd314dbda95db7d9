"""Seeded synthetic inputs for one PagedAttention step.

This module only draws numbers and lays them out in the op's input tensors:
packed new-token Q/K/V, a paged K/V pool whose past positions are filled, a
shuffled block table, cumulative/past sequence lengths and, for rotary runs,
the cos/sin tables.  It holds none of the attention, rotary or cache-write
arithmetic, so both the CUDA path and the CPU oracle can consume it.

Shapes follow the op contract of the CUDA PagedAttention design
("PagedAttention - CUDA Design Document", section 4 Schema and section 15
Validation Rules):

  query       [token_count, num_heads * head_size]        fp16
  key, value  [token_count, kv_num_heads * head_size]     fp16
  key_cache   [num_blocks, block_size, kv_num_heads, head_size] fp16 (NHD)
  block_table [batch, max_blocks_per_seq] int32, -1 = unmapped
  cumulative_sequence_lengths [batch + 1] int32
  past_sequence_lengths       [batch] int32
  cos_cache, sin_cache        [max_position, rotary_dim / 2] fp16

Pool contents: the slots holding positions [0, past_b) of every sequence are
N(0,1) fp16; every other slot (the new positions before the write, the 20 %
spare blocks, the tail of each last block) holds the fp16 NaN pattern
0x7E00, so a kernel that reads a slot it should not read produces NaN.

8-bit pools (quantized cache, CUDA design section 8): past slots hold random
codes (int8: a normal of standard deviation 32 drawn as integers and clipped
to +-127; e4m3fn: random sign, exponent field 0..10 and fraction bits, so
magnitudes up to 15), unused slots the code 0x80 (int8 -128, a loud value)
or 0x7F (e4m3fn NaN); k_scale / v_scale are fp32 [1] or [Hk*D], drawn
around 1/32 (int8) or 1/16 (e4m3fn).  head_sink is fp16 [H], N(0, 2^2).

bfloat16 steps (cache_dtype CACHE_BF16; the kernel is registered for fp16
and bfloat16 activations, CUDA design section 8.2): the same draws rounded to bfloat16 for
every 16-bit tensor (query, key, value, both pools, cos/sin, head_sink);
unused pool slots hold the bfloat16 NaN pattern 0x7FC0.  With act_bf16 an
8-bit step draws its activations the same way over the 8-bit pools above.
"""

from __future__ import annotations

import dataclasses
import math
from typing import Optional

import torch

NAN_SENTINEL_BITS = 0x7E00
BF16_NAN_SENTINEL_BITS = 0x7FC0


@dataclasses.dataclass(frozen=True)
class StepShape:
    """One workload: head geometry, paging geometry and the length recipe."""

    name: str
    num_heads: int
    kv_num_heads: int
    head_size: int
    block_size: int
    past_lens: tuple            # per sequence
    new_lens: tuple             # per sequence
    scale: float = 0.0          # 0 => 1/sqrt(head_size)
    softcap: float = 0.0
    local_window_size: int = -1
    do_rotary: int = 0
    rotary_interleaved: int = 0
    rotary_dim: int = 0         # 0 => head_size when do_rotary
    num_blocks: int = 0         # 0 => ceil(1.2 * blocks needed)
    max_blocks_per_seq: int = 0  # 0 => max over sequences of blocks needed
    seed: int = 0

    @property
    def batch(self) -> int:
        return len(self.past_lens)

    @property
    def token_count(self) -> int:
        return int(sum(self.new_lens))


def _blocks_needed(L: int, bs: int) -> int:
    return (L + bs - 1) // bs


def _lens_uniform(n, lo, hi, gen):
    return [int(x) for x in torch.randint(lo, hi + 1, (n,), generator=gen)]


def config_shape(index: int) -> StepShape:
    """The five named workloads (index 0..4).

    0 tiny mixed step; 1 Llama-3-8B-shaped decode; 2 mixed continuous-batch
    step (16 x 1024-token prefills + 240 decodes); 3 Gemma-2-shaped long
    decode with window 4096 and softcap 50; 4 Llama-70B-shaped decode with
    rotary.  Seeds: lengths use 3000+i, block shuffle 2000+i, values 1000+i.
    """
    lg = torch.Generator().manual_seed(3000 + index)
    if index == 0:
        return StepShape("tiny_mixed_b3_h4_kv2_d64_bs16", 4, 2, 64, 16,
                         (0, 17, 40), (5, 1, 1), scale=1.0 / 8.0,
                         num_blocks=64, max_blocks_per_seq=3, seed=index)
    if index == 1:
        past = _lens_uniform(64, 512, 4096, lg)
        return StepShape("llama3_8b_decode_b64_h32_kv8_d128_bs16", 32, 8, 128,
                         16, tuple(past), (1,) * 64, max_blocks_per_seq=257,
                         seed=index)
    if index == 2:
        dec_past = _lens_uniform(240, 1024, 8192, lg)
        past = [0] * 16 + dec_past
        new = [1024] * 16 + [1] * 240
        order = torch.randperm(256, generator=lg).tolist()
        past = [past[i] for i in order]
        new = [new[i] for i in order]
        return StepShape("mixed_16x1024_prefill_240_decode_h32_kv8_d128_bs32",
                         32, 8, 128, 32, tuple(past), tuple(new),
                         max_blocks_per_seq=257, seed=index)
    if index == 3:
        return StepShape("gemma2_long_decode_b8_h16_kv8_d256_bs64_w4096_cap50",
                         16, 8, 256, 64, (32768,) * 8, (1,) * 8,
                         scale=1.0 / 16.0, softcap=50.0,
                         local_window_size=4096, max_blocks_per_seq=513,
                         seed=index)
    if index == 4:
        z = torch.randn(256, generator=lg, dtype=torch.float64)
        past = torch.exp(math.log(2048.0) + 1.0 * z).round().clamp(1, 16384)
        return StepShape("llama70b_rotary_decode_b256_h64_kv8_d128_bs16",
                         64, 8, 128, 16, tuple(int(x) for x in past),
                         (1,) * 256, do_rotary=1, max_blocks_per_seq=1025,
                         seed=index)
    raise ValueError(f"no workload {index}")


def custom_shape(name, num_heads, kv_num_heads, head_size, block_size,
                 past_lens, new_lens, seed=7, **kw) -> StepShape:
    return StepShape(name, num_heads, kv_num_heads, head_size, block_size,
                     tuple(int(x) for x in past_lens),
                     tuple(int(x) for x in new_lens), seed=seed, **kw)


def _fill_sentinel(t: torch.Tensor) -> torch.Tensor:
    pattern = BF16_NAN_SENTINEL_BITS if t.dtype == torch.bfloat16 else NAN_SENTINEL_BITS
    return t.view(torch.int16).fill_(pattern).view(t.dtype)


CACHE_FP16, CACHE_INT8, CACHE_FP8, CACHE_BF16 = 0, 1, 2, 3
QUANT_NONE, QUANT_PER_TENSOR, QUANT_PER_CHANNEL = 0, 1, 2


def make_step(shape: StepShape, device="cpu", gen_device: Optional[str] = None,
              cache_dtype: int = CACHE_FP16, quant_type: int = QUANT_NONE,
              head_sink: bool = False, qk_norm: bool = False, packed_qkv: bool = False,
              latent_v_head_size: int = 0, act_bf16: bool = False):
    """Build every input tensor of one step on `device`.

    Random values are drawn with a torch.Generator on `gen_device` (default:
    `device`), so a CPU run and a CUDA run of the same shape share lengths
    and block tables (drawn on the CPU) but not necessarily values.
    cache_dtype / quant_type select 8-bit pools with their scales, or
    (CACHE_BF16) bfloat16 activations and pools; act_bf16 with an 8-bit
    cache_dtype makes the activations bfloat16 over 8-bit pools; head_sink
    adds a per-head sink input; qk_norm adds q/k norm weights ([D] fp16 or
    bfloat16, 1 + 0.3 N(0,1)); packed_qkv lays Q, K and V out as one [T, (H+2Hk)*D]
    query tensor with key and value None.  latent_v_head_size > 0 makes a
    multi-head latent attention step (CUDA design section 12): one kv head,
    key rows of head_size latent channels, value and value_cache None, V the
    first latent_v_head_size channels, rotary (if on) over the last
    rotary_dim channels.
    """
    gen_device = gen_device or str(device)
    H, Hk, D, bs = shape.num_heads, shape.kv_num_heads, shape.head_size, shape.block_size
    B = shape.batch
    past = list(shape.past_lens)
    new = list(shape.new_lens)
    L = [p + n for p, n in zip(past, new)]
    need = [_blocks_needed(x, bs) for x in L]
    MB = shape.max_blocks_per_seq or max(max(need), 1)
    if max(need, default=0) > MB:
        raise ValueError("max_blocks_per_seq too small for the lengths")
    NB = shape.num_blocks or max(1, math.ceil(1.2 * sum(need)))
    if sum(need) > NB:
        raise ValueError("pool too small")

    bg = torch.Generator().manual_seed(2000 + shape.seed)
    perm = torch.randperm(NB, generator=bg)
    bt = torch.full((B, MB), -1, dtype=torch.int32)
    cur = 0
    for b in range(B):
        bt[b, :need[b]] = perm[cur:cur + need[b]].to(torch.int32)
        cur += need[b]

    cum = torch.zeros(B + 1, dtype=torch.int32)
    cum[1:] = torch.cumsum(torch.tensor(new, dtype=torch.int64), 0).to(torch.int32)
    T = int(cum[-1])

    vg = torch.Generator(device=gen_device).manual_seed(1000 + shape.seed)
    if act_bf16 and cache_dtype not in (CACHE_INT8, CACHE_FP8):
        raise ValueError("act_bf16 goes with an 8-bit cache (CACHE_BF16 is the 16-bit form)")
    act = torch.bfloat16 if cache_dtype == CACHE_BF16 or act_bf16 else torch.float16

    def randn(*size):
        return torch.randn(*size, generator=vg, device=gen_device,
                           dtype=torch.float32).to(act).to(device)

    query = randn(T, H * D)
    key = randn(T, Hk * D)
    value = randn(T, Hk * D)

    if cache_dtype in (CACHE_FP16, CACHE_BF16):
        key_cache = _fill_sentinel(torch.empty(NB, bs, Hk, D, dtype=act, device=device))
        value_cache = _fill_sentinel(torch.empty(NB, bs, Hk, D, dtype=act, device=device))
        draw = randn
    else:
        fill = 0x80 if cache_dtype == CACHE_INT8 else 0x7F
        key_cache = torch.full((NB, bs, Hk, D), fill, dtype=torch.uint8, device=device)
        value_cache = torch.full((NB, bs, Hk, D), fill, dtype=torch.uint8, device=device)

        def draw(*size):
            if cache_dtype == CACHE_INT8:
                v = torch.randn(*size, generator=vg, device=gen_device).mul(32.0).round().clamp(-127, 127)
                return v.to(torch.int8).view(torch.uint8).to(device)
            sign = torch.randint(0, 2, size, generator=vg, device=gen_device)
            expo = torch.randint(0, 11, size, generator=vg, device=gen_device)
            frac = torch.randint(0, 8, size, generator=vg, device=gen_device)
            return (sign * 128 + expo * 8 + frac).to(torch.uint8).to(device)
    # Past content, laid out block by block: row i of a sequence's block table
    # names the block holding its positions [i*bs, (i+1)*bs).
    for b in range(B):
        full, rem = divmod(past[b], bs)
        if full:
            ids = bt[b, :full].to(torch.int64).to(device)
            key_cache[ids] = draw(full, bs, Hk, D)
            value_cache[ids] = draw(full, bs, Hk, D)
        if rem:
            blk = int(bt[b, full])
            key_cache[blk, :rem] = draw(rem, Hk, D)
            value_cache[blk, :rem] = draw(rem, Hk, D)

    out = dict(
        query=query, key=key, value=value,
        key_cache=key_cache, value_cache=value_cache,
        block_table=bt.to(device),
        cumulative_sequence_lengths=cum.to(device),
        past_sequence_lengths=torch.tensor(past, dtype=torch.int32).to(device),
        batch=B, token_count=T, num_heads=H, kv_num_heads=Hk, head_size=D,
        block_size=bs, num_blocks=NB, max_blocks_per_seq=MB,
        scale=shape.scale, softcap=shape.softcap,
        local_window_size=shape.local_window_size,
        do_rotary=shape.do_rotary, rotary_interleaved=shape.rotary_interleaved,
        cos_cache=None, sin_cache=None, rotary_dim=0,
    )
    if shape.do_rotary:
        R = shape.rotary_dim or D
        cos, sin = rotary_tables(MB * bs, R, dtype=act)
        out.update(cos_cache=cos.to(device), sin_cache=sin.to(device), rotary_dim=R)
    if cache_dtype == CACHE_BF16:
        out.update(cache_dtype=cache_dtype)
    elif cache_dtype != CACHE_FP16:
        sg = torch.Generator().manual_seed(4000 + shape.seed)
        n = Hk * D if quant_type == QUANT_PER_CHANNEL else 1
        base = 1.0 / 32.0 if cache_dtype == CACHE_INT8 else 1.0 / 16.0
        ks = base * (0.8 + 0.4 * torch.rand(n, generator=sg))
        vs = base * (0.8 + 0.4 * torch.rand(n, generator=sg))
        out.update(cache_dtype=cache_dtype, quant_type=quant_type,
                   k_scale=ks.float().to(device), v_scale=vs.float().to(device))
        if act_bf16:
            out.update(act_bf16=True)
    if head_sink:
        hg = torch.Generator().manual_seed(5000 + shape.seed)
        out.update(head_sink=(2.0 * torch.randn(H, generator=hg)).to(act).to(device))
    if qk_norm:
        ng = torch.Generator().manual_seed(6000 + shape.seed)
        out.update(q_norm_weight=(1.0 + 0.3 * torch.randn(D, generator=ng)).to(act).to(device),
                   k_norm_weight=(1.0 + 0.3 * torch.randn(D, generator=ng)).to(act).to(device),
                   qk_norm_epsilon=1e-6)
    if packed_qkv:
        out.update(query=torch.cat([out["query"], out["key"], out["value"]], dim=1).contiguous(),
                   key=None, value=None)
    if latent_v_head_size:
        if Hk != 1:
            raise ValueError("a latent cache has one kv head")
        out.update(value=None, value_cache=None, kv_cache_layout=1, v_head_size=latent_v_head_size,
                   rotary_offset=(D - (out["rotary_dim"] or 0)) if shape.do_rotary else 0)
    return out


def rotary_tables(max_position: int, rotary_dim: int, base: float = 10000.0, dtype=torch.float16):
    """cos/sin tables [max_position, rotary_dim/2] as fp16 (or `dtype`).

    theta_i = base^(-2i/rotary_dim); entry (p, i) = cos/sin(p * theta_i),
    evaluated in fp64 and rounded to the table type.  These are op inputs (the model's
    rotary cache), not part of the op.
    """
    half = rotary_dim // 2
    i = torch.arange(half, dtype=torch.float64)
    inv = base ** (-2.0 * i / rotary_dim)
    ang = torch.arange(max_position, dtype=torch.float64)[:, None] * inv[None, :]
    return torch.cos(ang).to(dtype), torch.sin(ang).to(dtype)

