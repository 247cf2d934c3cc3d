"""Turns the hand-worked cases in tests/golden/decode_examples.json into arrays
in the library's layouts.  Values are encoded with numpy (f16) or by taking the
upper half of the float32 (bf16; every fixture value is exact in bf16)."""
import json
import math
import os
from fractions import Fraction

import numpy as np

PATH = os.path.join(os.path.dirname(__file__), "golden", "decode_examples.json")


def load():
    return json.load(open(PATH))


def enc16(x, dtype):
    x = np.asarray(x, dtype=np.float64)
    if dtype == "f16":
        h = x.astype(np.float16)
        assert np.array_equal(h.astype(np.float64), x), "fixture value not exact in f16"
        return h.view(np.uint16)
    f = x.astype(np.float32)
    b = (f.view(np.uint32) >> 16).astype(np.uint16)
    assert np.array_equal((b.astype(np.uint32) << 16).view(np.float32).astype(np.float64), x), \
        "fixture value not exact in bf16"
    return b


def scalar(v):
    if isinstance(v, (int, float)):
        return float(v)
    v = v.strip()
    if v.endswith("ln2"):
        k = v[:-3] or "1"
        return float(k) * math.log(2.0)
    return float(Fraction(v))


def case_arrays(c):
    """Returns dict(q, k_cache, v_cache, block_tables, context_lens, scale, kv_scale, expected)."""
    NB, bs, Hq, Hkv, D = c["num_blocks"], c["block_size"], c["num_q_heads"], c["num_kv_heads"], c["head_dim"]
    q = enc16(np.array(c["q"], np.float64), c["dtype"])
    if c["kv_dtype"] == "fp8":
        kc = np.zeros((NB, Hkv, bs, D), np.uint8)
        vc = np.zeros((NB, Hkv, bs, D), np.uint8)
        for t in c["fp8_tokens"]:
            b, o = divmod(t["slot"], bs)
            kc[b, :, o, :] = np.array([[int(x, 16) for x in row] for row in t["k_codes"]], np.uint8)
            vc[b, :, o, :] = np.array([[int(x, 16) for x in row] for row in t["v_codes"]], np.uint8)
    else:
        fill = np.full((NB, Hkv, bs, D), float(c.get("fill", 0.0)))
        kf, vf = fill.copy(), fill.copy()
        for t in c["tokens"]:
            b, o = divmod(t["slot"], bs)
            kf[b, :, o, :] = np.array(t["k"], np.float64)
            vf[b, :, o, :] = np.array(t["v"], np.float64)
        kc, vc = enc16(kf, c["kv_dtype"]), enc16(vf, c["kv_dtype"])
    exp = np.array([[[float(Fraction(x)) for x in row] for row in seq] for seq in c["expected"]], np.float64)
    return dict(q=q, k_cache=kc, v_cache=vc,
                block_tables=np.array(c["block_tables"], np.int32),
                context_lens=np.array(c["context_lens"], np.int32),
                scale=scalar(c["scale"]), kv_scale=float(c["kv_scale"]), expected=exp)
