"""Pins for the oracle's explicit slot_mapping write and the rolling
(ring-buffer) sliding-window cache ("PagedAttention - CUDA Design Document",
sections 5.2 and 9.3), each against something other than the oracle:

  * slot_mapping = the hand-derived slots of tests/golden/cache_write_slots.txt
    gives the pool of the derived write (pinned by that golden file), with
    "none" rows passed as -1
  * -1 skips exactly that row; a slot outside every table row is written
    there (the definition: slot_mapping is authoritative for writes)
  * ring buffer: a sequence held in N = ceil(W / bs) + 1 recycled blocks,
    table entries below the live range -1, gives the same attention as the
    full cache with the same window, over several decode steps (section
    9.3.5); with W >= L the ring never recycles and equals full attention
"""

import math

import numpy as np
import torch

import oracle
from test_oracle_pins import SENT, _parse_golden, bits, h16


def _golden_case():
    meta, rows = _parse_golden("tests/golden/cache_write_slots.txt")
    bs, NB = meta["block_size"][0], meta["num_blocks"][0]
    Hk, D = meta["kv_num_heads"][0], meta["head_size"][0]
    bt = torch.tensor(meta["block_table"], dtype=torch.int32)
    past = torch.tensor(meta["past"], dtype=torch.int32)
    cum = torch.tensor([0] + list(np.cumsum(meta["new"])), dtype=torch.int32)
    T = int(cum[-1])
    key = h16(np.repeat(np.arange(1, T + 1, dtype=np.float32)[:, None], Hk * D, 1))
    return bs, NB, Hk, D, bt, past, cum, T, key, rows


def test_slot_mapping_equal_to_golden_slots_gives_the_derived_pool():
    bs, NB, Hk, D, bt, past, cum, T, key, rows = _golden_case()
    slots = np.array([-1 if r[5] == "none" else int(r[5]) for r in rows], dtype=np.int32)
    pool = np.full((NB, bs, Hk, D), SENT, dtype=np.uint16)
    dk, dv = oracle.cache_write(bits(key), bits(-key), pool, pool, bt, cum, past, Hk, D, bs)
    ek, ev = oracle.cache_write(bits(key), bits(-key), pool, pool, bt, cum, past, Hk, D, bs, slot_mapping=slots)
    assert np.array_equal(dk, ek) and np.array_equal(dv, ev)


def test_slot_mapping_minus_one_skips_and_other_slots_are_written():
    bs, NB, Hk, D, bt, past, cum, T, key, rows = _golden_case()
    pool = np.full((NB, bs, Hk, D), SENT, dtype=np.uint16)
    # token 0 -> slot 100 (block 6, in no table row), token 1 skipped, others 0..3
    slots = np.array([100, -1, 0, 1, 2, 3], dtype=np.int32)
    kc, vc = oracle.cache_write(bits(key), bits(-key), pool, pool, bt, cum, past, Hk, D, bs, slot_mapping=slots)
    kf = kc.reshape(NB * bs, Hk * D).view(np.float16)
    written = {100: 1, 0: 3, 1: 4, 2: 5, 3: 6}
    for s in range(NB * bs):
        if s in written:
            assert np.all(kf[s] == written[s])
        else:
            assert np.all(kc.reshape(NB * bs, Hk * D)[s] == SENT)
    bad = np.array([100, -2, 0, 1, 2, 3], dtype=np.int32)
    try:
        oracle.cache_write(bits(key), bits(-key), pool, pool, bt, cum, past, Hk, D, bs, slot_mapping=bad)
        raise AssertionError("out-of-range slot accepted")
    except ValueError:
        pass


def _ring_run(L0, steps, W, bs, H, Hk, D, seed):
    """Full-cache and ring-cache attention of one decode sequence per step."""
    g = torch.Generator().manual_seed(seed)
    Lmax = L0 + steps
    Kd = torch.randn(Lmax, Hk, D, generator=g).half()
    Vd = torch.randn(Lmax, Hk, D, generator=g).half()
    MB = math.ceil(Lmax / bs)
    N = math.ceil(W / bs) + 1
    full_nb = MB
    full_k = np.full((full_nb, bs, Hk, D), SENT, np.uint16)
    full_v = full_k.copy()
    bt_full = torch.arange(MB, dtype=torch.int32)[None, :]
    ring = np.arange(full_nb, full_nb + N)  # ring blocks live in a pool of their own
    ring_k = np.full((full_nb + N, bs, Hk, D), SENT, np.uint16)
    ring_v = ring_k.copy()
    for p in range(L0):  # past content
        full_k[p // bs, p % bs] = bits(Kd[p])
        full_v[p // bs, p % bs] = bits(Vd[p])
        i = p // bs
        ring_k[ring[i % N], p % bs] = bits(Kd[p])
        ring_v[ring[i % N], p % bs] = bits(Vd[p])
    outs = []
    for s in range(steps):
        p = L0 + s
        cum = torch.tensor([0, 1], dtype=torch.int32)
        past = torch.tensor([p], dtype=torch.int32)
        q = torch.randn(1, H * D, generator=g).half()
        # full cache: derived write
        full_k, full_v = oracle.cache_write(bits(Kd[p].reshape(1, -1)), bits(Vd[p].reshape(1, -1)), full_k, full_v,
                                            bt_full, cum, past, Hk, D, bs)
        # ring: explicit slot, live table entries point into the ring, older ones -1
        i = p // bs
        slot = np.array([ring[i % N] * bs + p % bs], dtype=np.int32)
        ring_k, ring_v = oracle.cache_write(bits(Kd[p].reshape(1, -1)), bits(Vd[p].reshape(1, -1)), ring_k, ring_v,
                                            bt_full, cum, past, Hk, D, bs, slot_mapping=slot)
        live0 = max(0, p - W + 1) // bs
        bt_ring = torch.full((1, MB), -1, dtype=torch.int32)
        for j in range(live0, i + 1):
            bt_ring[0, j] = int(ring[j % N])
        a = oracle.attention(bits(q), full_k, full_v, bt_full, cum, past, H, Hk, D, bs, 0.0, 0.0, W)
        b = oracle.attention(bits(q), ring_k, ring_v, bt_ring, cum, past, H, Hk, D, bs, 0.0, 0.0, W)
        outs.append((a, b))
    return outs


def test_ring_buffer_cache_equals_full_cache():
    for (a, b) in _ring_run(L0=70, steps=40, W=33, bs=16, H=4, Hk=2, D=16, seed=3):
        assert np.array_equal(a, b)


def test_ring_buffer_with_window_beyond_context_is_full_attention():
    outs = _ring_run(L0=20, steps=5, W=64, bs=16, H=4, Hk=2, D=16, seed=4)
    # with W >= L every position stays live: the ring run equals the full run
    for (a, b) in outs:
        assert np.array_equal(a, b)
