"""Strength of the oracle's pins: each plausible mistake below is planted in
a copy of oracle.c (on the CPU, never in the library under test), the copy
is compiled, and the oracle pin tests are run against it in a child
process.  Every mutant must make at least one pin fail; the unmodified copy
must pass them all.

The mistakes are the ones an implementation of the pages' formulas could
plausibly make: the GQA head map, the causal and window bounds, softcap
without its outer factor, the default 1/sqrt(D) scale, the head_sink term,
the sign and pairing of the rotation and its channel offset, the slot
derivation, the binary16 and e4m3fn roundings, int8 rounding and
clipping, the per-channel scale index, the QK-Norm epsilon, weight and the
order and precision of its sum of squares, the latent layout (scores over
all 576 channels, values from the first 512), and the bfloat16 paths
(decode exponent, rounding, bfloat16 read as fp16, rotary rounded to fp16,
bfloat16 activations over an 8-bit cache quantized or attended as fp16).
"""

import os
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "oracle.c")
PIN_FILES = [os.path.join(ROOT, "tests", f) for f in (
    "test_oracle_pins.py", "test_oracle_quant_pins.py", "test_oracle_slot_pins.py",
    "test_oracle_qknorm_pins.py", "test_oracle_mla_pins.py", "test_oracle_bf16_pins.py",
    "test_oracle_bf16_quant_pins.py")]

# (name, text in oracle.c, replacement, occurrences of the text, indices replaced or None = all)
MUTANTS = [
    ("gqa head map h % Hk", "int k = h / G;", "int k = h % Hk;", 1, None),
    ("gqa causal bound", "int kv_len = pos + 1;", "int kv_len = pos;", 2, (0,)),
    ("latent causal bound", "int kv_len = pos + 1;", "int kv_len = pos + 2;", 2, (1,)),
    ("gqa window bound", "lo = kv_len - window;", "lo = kv_len - window + 1;", 1, None),
    ("latent window bound", "? kv_len - window : 0;", "? kv_len - window - 1 : 0;", 1, None),
    ("gqa softcap outer factor", "x = softcap * tanh(x / softcap);", "x = tanh(x / softcap);", 4, (0, 1)),
    ("latent softcap outer factor", "x = softcap * tanh(x / softcap);", "x = tanh(x / softcap);", 4, (2, 3)),
    ("default scale 1/D", "scale = 1.0 / sqrt((double)D);", "scale = 1.0 / (double)D;", 1, None),
    ("sink term without the max", "denom += exp(sink - xmax);", "denom += exp(sink);", 1, None),
    ("rotary sign", "float y1 = t1 - t2;", "float y1 = t1 + t2;", 1, None),
    ("rotary pairing", "i + half_rot);", "i + half_rot - 1);", 1, None),
    ("rotary offset ignored", "int i1 = offset + (interleaved", "int i1 = (interleaved", 1, None),
    ("slot offset", "return (long long)blk * bs + pos % bs;", "return (long long)blk * bs + (pos + 1) % bs;", 1,
     None),
    ("binary16 truncation", "double m = nearbyint(ldexp(a, 11 - e));", "double m = floor(ldexp(a, 11 - e));", 1,
     None),
    ("binary16 subnormal exponent", "v = ldexp((double)f, -24);", "v = ldexp((double)f, -25);", 1, None),
    ("e4m3fn NaN instead of saturation", "if (a >= 448.0) return sign | 0x7e;", "if (a >= 448.0) return sign | 0x7f;",
     1, None),
    ("e4m3fn truncation", "double m = nearbyint(ldexp(a, 4 - e));", "double m = floor(ldexp(a, 4 - e));", 1, None),
    ("int8 truncation", "float r = nearbyintf(y);", "float r = truncf(y);", 1, None),
    ("int8 without the upper clip", "if (r > 127.0f) r = 127.0f;", "", 1, None),
    ("per-channel scale index", "k_scale[per_channel ? k * D + c : 0]", "k_scale[per_channel ? c : 0]", 2, None),
    ("K quantized with the V scale", "oracle_quantize(key[(size_t)t * row + e], k_scale[si]",
     "oracle_quantize(key[(size_t)t * row + e], v_scale[si]", 1, None),
    ("QK-Norm without epsilon", "float v = mean + eps;", "float v = mean;", 1, None),
    ("QK-Norm without weight", "float b = a * (float)elem16_to_double(w[c], bf16);", "float b = a;", 1, None),
    ("QK-Norm sum from the last channel", "for (int c = 0; c < D; ++c) {\n        float v = (float)elem16_to_double(xr[c], bf16);",
     "for (int c = D - 1; c >= 0; --c) {\n        float v = (float)elem16_to_double(xr[c], bf16);", 1, None),
    ("bfloat16 QK-Norm rounded to fp16", "tmp[c] = bf16 ? oracle_double_to_bf16((double)b)",
     "tmp[c] = 0 ? oracle_double_to_bf16((double)b)", 1, None),
    ("QK-Norm sum in fp64", "float sum = 0.0f;", "double sum = 0.0;", 1, None),
    ("latent V from the last channels", "o[c] += w * oracle_half_to_double(lr[c]);",
     "o[c] += w * oracle_half_to_double(lr[c + D - Dv]);", 1, None),
    ("latent scores over the V channels only", "for (int c = 0; c < D; ++c) x += q[c] * oracle_half_to_double(lr[c]);",
     "for (int c = 0; c < Dv; ++c) x += q[c] * oracle_half_to_double(lr[c]);", 2, None),
    ("bfloat16 exponent bias", "v = ldexp((double)(128 + f), e - 134);", "v = ldexp((double)(128 + f), e - 133);",
     1, None),
    ("bfloat16 truncation", "double m = nearbyint(ldexp(a, 8 - e));", "double m = floor(ldexp(a, 8 - e));", 1,
     None),
    ("bfloat16 query read as fp16", "q[c] = elem16_to_double(query[((size_t)t * H + h) * D + c], bf16);",
     "q[c] = oracle_half_to_double(query[((size_t)t * H + h) * D + c]);", 1, None),
    ("bfloat16 sink read as fp16", "elem16_to_double(head_sink[h], bf16)", "oracle_half_to_double(head_sink[h])", 1,
     None),
    ("bfloat16 activations quantized as fp16", "(float)elem16_to_double(h, (cache_dtype & ORACLE_ACT_BF16) != 0) / s",
     "(float)elem16_to_double(h, 0) / s", 1, None),
    ("bfloat16 activations over 8-bit pools attended as fp16",
     "cache_dtype == ORACLE_CACHE_BF16 || (cache_dtype & ORACLE_ACT_BF16) != 0;",
     "cache_dtype == ORACLE_CACHE_BF16;", 1, None),
    ("bfloat16 rotary rounded to fp16", "tmp[i1] = bf16 ? oracle_double_to_bf16((double)y1)",
     "tmp[i1] = 0 ? oracle_double_to_bf16((double)y1)", 1, None),
]


def _mutate(text, old, new, count, which):
    parts = text.split(old)
    assert len(parts) - 1 == count, f"oracle.c holds {len(parts) - 1} copies of {old!r}, expected {count}"
    out = parts[0]
    for i, rest in enumerate(parts[1:]):
        out += (new if which is None or i in which else old) + rest
    return out


def _run_pins(directory, text):
    os.makedirs(directory, exist_ok=True)
    src = os.path.join(directory, "oracle.c")
    with open(src, "w") as f:
        f.write(text)
    lib = os.path.join(directory, "liboracle.so")
    cc = subprocess.run(["gcc", "-O2", "-ffp-contract=off", "-fno-fast-math", "-std=c11", "-shared", "-fPIC",
                         "-o", lib, src, "-lm"], capture_output=True, text=True)
    if cc.returncode != 0:
        return "compile", cc.stderr[-2000:]
    env = dict(os.environ, PA_ORACLE_SOURCE=src)
    r = subprocess.run([sys.executable, "-m", "pytest", "-x", "-q", "-m", "not gpu", "-p", "no:cacheprovider",
                        *PIN_FILES], cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    return r.returncode, r.stdout[-3000:] + r.stderr[-2000:]


def test_every_planted_mistake_fails_a_pin(tmp_path):
    text = open(SRC).read()
    jobs = [("unmodified", str(tmp_path / "unmodified"), text)]
    for i, (name, old, new, count, which) in enumerate(MUTANTS):
        jobs.append((name, str(tmp_path / f"m{i:02d}"), _mutate(text, old, new, count, which)))
    with ThreadPoolExecutor(max_workers=min(8, os.cpu_count() or 1)) as ex:
        results = list(ex.map(lambda j: _run_pins(j[1], j[2]), jobs))
    rc0, out0 = results[0]
    assert rc0 == 0, f"the unmodified oracle fails its pins:\n{out0}"
    survivors = []
    for (name, _, _), (rc, out) in zip(jobs[1:], results[1:]):
        if rc == "compile":
            pytest.fail(f"mutant '{name}' does not compile:\n{out}")
        if rc != 1 or "failed" not in out:
            survivors.append(f"{name} (exit {rc})")
    assert not survivors, "mistakes no pin catches: " + ", ".join(survivors)
