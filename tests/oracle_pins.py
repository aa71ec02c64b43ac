"""Pins that tie the fp64 oracle to facts outside itself.

Each ``pin_*`` takes a decode function with the signature of
``oracle.mla_decode`` and raises ``AssertionError`` when the function breaks a
fact that the mathematics (or a page's worked definition) fixes:

  pin_brute_force        unpaged brute force on tiny inputs (plain exp/sum, no
                         max shift, matrix form over contiguous rows)
  pin_permutation        moving physical pages and rewriting block_table does
                         not change a single bit of the result
  pin_q_zero             q = 0: O is the mean of the visible V rows, LSE = ln T
  pin_seqlen_one         one key: O is that key's V row, LSE = scale * q.k
  pin_two_key_golden     hand-derived two-key example (tests/golden/two_key.txt)
  pin_score_shift        a common RoPE part in every key shifts all scores by
                         one constant: O unchanged, LSE shifted by it
  pin_causal_consistency query i of a causal multi-token call equals a
                         one-token call over seqlen - s_q + i + 1 keys
  pin_zero_visible       rows with no visible key: O = 0, LSE = -inf
  pin_kv_head_groups     with h_kv > 1, head h reads KV head h // (h_q / h_kv)
  pin_sampled_rows       the row-subset entry point equals the full call
  pin_saturated_softmax  one key's score exceeds the others by ~1000: O is that
                         key's V row and LSE its score (needs the max shift)

Pins of the packed e4m3 cache (``FP8_PINS``; they take the bf16 decode, the
e4m3 decode and the oracle's e4m3 code decoder):

  pin_e4m3_codes         all 256 codes against torch's float8_e4m3fn decoding
                         (a library routine) and the OCP E4M3 landmarks
  pin_fp8_matches_bf16   with power-of-two scales every dequantized value is a
                         bf16 value: the e4m3 decode must then equal, bit for
                         bit, the bf16 decode of the dequantized cache
  pin_fp8_scale_linearity  doubling every token's scale and halving q leaves
                         the scores unchanged and doubles O exactly

Pins of the sparse top-k decode (``SPARSE_PINS``; they take the dense and the
sparse decode):

  pin_sparse_brute_force   numpy gather-and-softmax over each query token's
                           list (entries outside [0, T) dropped, repeats kept)
  pin_sparse_full_list     the list 0 .. T-1 (padded with -1) gives the dense
                           decode bit for bit
  pin_sparse_order         permuting a list changes nothing beyond rounding;
                           appending ignored entries changes no bit

The mutation test in ``test_oracle_pins.py`` plants mistakes in a copy of the
oracle's C source and checks that some pin catches each one.
"""
from __future__ import annotations

import math
import os

import numpy as np
import torch

GOLDEN_DIR = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


# ---------------------------------------------------------------- input helpers
def bf16_bits_of(x) -> np.ndarray:
    """Round fp32/fp64 values to bf16 (nearest even) and return the uint16 bits."""
    t = torch.as_tensor(np.asarray(x, dtype=np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16).copy()


def f64_of(bits) -> np.ndarray:
    """Exact fp64 value of bf16 bit patterns (through torch's own conversion)."""
    t = torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16)
    return t.to(torch.float64).numpy()


def rand_bits(rng, shape, scale=1.0):
    return bf16_bits_of(rng.standard_normal(shape) * scale)


def page_out(rows_per_seq, page, rng, extra_pages=1, garbage=1e4):
    """Scatter contiguous per-sequence rows [T_b, h_kv, d] (bf16 bits) into a paged pool.

    Returns (kcache bits [pool, page, h_kv, d], block_table int32 [b, max_blocks]).
    Unused rows and pages hold large finite garbage.
    """
    h_kv, d = rows_per_seq[0].shape[1:]
    n_pages = [(r.shape[0] + page - 1) // page for r in rows_per_seq]
    max_blocks = max(1, max(n_pages))
    pool = sum(n_pages) + extra_pages
    kc = rand_bits(rng, (pool, page, h_kv, d), scale=garbage)
    perm = rng.permutation(pool).astype(np.int32)
    bt = rng.integers(0, pool, size=(len(rows_per_seq), max_blocks)).astype(np.int32)
    cur = 0
    for b, rows in enumerate(rows_per_seq):
        for p in range(n_pages[b]):
            phys = perm[cur]
            cur += 1
            bt[b, p] = phys
            chunk = rows[p * page:(p + 1) * page]
            kc[phys, :chunk.shape[0]] = chunk
    return kc, bt


def visible(seqlen, s_q, i, causal):
    return seqlen - s_q + i + 1 if causal else seqlen


# ---------------------------------------------------------------- pins
def _brute(q_bits, rows_per_seq, seqlens, dv, scale, causal, h_kv):
    qf = f64_of(q_bits)
    b, s_q, h_q, d = qf.shape
    o = np.zeros((b, s_q, h_q, dv))
    lse = np.zeros((b, s_q, h_q))
    for bi in range(b):
        kf = f64_of(rows_per_seq[bi])                      # [T, h_kv, d]
        for i in range(s_q):
            T = visible(int(seqlens[bi]), s_q, i, causal)
            for h in range(h_q):
                g = h // (h_q // h_kv)
                if T <= 0:
                    lse[bi, i, h] = -math.inf
                    continue
                K = kf[:T, g, :]
                e = np.exp(scale * (K @ qf[bi, i, h]))
                o[bi, i, h] = (e @ K[:, :dv]) / e.sum()
                lse[bi, i, h] = math.log(e.sum())
    return o, lse


def pin_brute_force(decode, seed=11):
    rng = np.random.default_rng(seed)
    cases = [
        # (b, s_q, h_q, h_kv, seqlens, causal, d, dv, page)
        (2, 1, 16, 1, [100, 37], False, 576, 512, 64),
        (3, 1, 4, 1, [1, 64, 200], False, 576, 512, 64),
        (2, 3, 4, 1, [5, 130], True, 576, 512, 64),
        (2, 2, 4, 2, [70, 3], False, 576, 512, 64),
        (2, 2, 8, 1, [130, 65], True, 512, 512, 64),    # the 512-wide row: V is the whole row
        (1, 4, 2, 1, [9], True, 40, 24, 4),
    ]
    for (b, s_q, h_q, h_kv, seqlens, causal, d, dv, page) in cases:
        q = rand_bits(rng, (b, s_q, h_q, d))
        rows = [rand_bits(rng, (T, h_kv, d)) for T in seqlens]
        kc, bt = page_out(rows, page, rng)
        scale = 1.0 / math.sqrt(d)
        o, lse = decode(q, kc, bt, np.array(seqlens, np.int32), dv, scale, causal)
        o_ref, lse_ref = _brute(q, rows, seqlens, dv, scale, causal, h_kv)
        assert np.allclose(lse, lse_ref, rtol=0, atol=1e-11), "LSE differs from brute force"
        assert np.allclose(o, o_ref, rtol=1e-11, atol=1e-12), "O differs from brute force"


def pin_permutation(decode, seed=12):
    rng = np.random.default_rng(seed)
    seqlens = [150, 64, 1, 129]
    d, dv, page = 576, 512, 64
    q = rand_bits(rng, (4, 2, 8, d))
    rows = [rand_bits(rng, (T, 1, d)) for T in seqlens]
    kc, bt = page_out(rows, page, rng, extra_pages=3)
    sl = np.array(seqlens, np.int32)
    o1, l1 = decode(q, kc, bt, sl, dv, 1 / 24, True)
    perm = rng.permutation(kc.shape[0])
    kc2 = np.empty_like(kc)
    kc2[perm] = kc
    bt2 = perm[bt].astype(np.int32)
    o2, l2 = decode(q, kc2, bt2, sl, dv, 1 / 24, True)
    assert np.array_equal(o1, o2) and np.array_equal(l1, l2), "result depends on physical page placement"


def pin_q_zero(decode, seed=13):
    rng = np.random.default_rng(seed)
    seqlens = [7, 64, 65, 300]
    d, dv, page, s_q = 576, 512, 64, 3
    q = bf16_bits_of(np.zeros((4, s_q, 4, d)))
    rows = [rand_bits(rng, (T, 1, d)) for T in seqlens]
    kc, bt = page_out(rows, page, rng)
    for causal in (False, True):
        o, lse = decode(q, kc, bt, np.array(seqlens, np.int32), dv, 1 / 24, causal)
        for b, T0 in enumerate(seqlens):
            vf = f64_of(rows[b])[:, 0, :dv]
            for i in range(s_q):
                T = visible(T0, s_q, i, causal)
                assert abs(lse[b, i, 0] - math.log(T)) < 1e-12, "LSE(q=0) != ln T"
                assert np.allclose(o[b, i], vf[:T].mean(axis=0), rtol=1e-12, atol=1e-13), "O(q=0) != mean V"


def pin_seqlen_one(decode, seed=14):
    rng = np.random.default_rng(seed)
    d, dv = 576, 512
    q = rand_bits(rng, (3, 1, 4, d))
    rows = [rand_bits(rng, (1, 1, d)) for _ in range(3)]
    kc, bt = page_out(rows, 64, rng)
    scale = 1 / 24
    o, lse = decode(q, kc, bt, np.array([1, 1, 1], np.int32), dv, scale, False)
    for b in range(3):
        v = f64_of(rows[b])[0, 0]
        for h in range(4):
            exact = scale * math.fsum(f64_of(q)[b, 0, h] * v)
            assert abs(lse[b, 0, h] - exact) < 1e-12, "LSE(one key) != scale*q.k"
            assert np.array_equal(o[b, 0, h], v[:dv]), "O(one key) != V row"


def load_two_key_golden():
    path = os.path.join(GOLDEN_DIR, "two_key.txt")
    vals = {}
    with open(path) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if not line:
                continue
            key, rest = line.split("=", 1)
            vals[key.strip()] = [float(x) for x in rest.split()]
    return vals


def pin_two_key_golden(decode):
    g = load_two_key_golden()
    d, dv, page = int(g["d"][0]), int(g["dv"][0]), int(g["page"][0])
    q = bf16_bits_of(np.array(g["q"]).reshape(1, 1, 1, d))
    kc = bf16_bits_of(np.array(g["kcache"]).reshape(-1, page, 1, d))
    bt = np.array(g["block_table"], np.int32).reshape(1, -1)
    o, lse = decode(q, kc, bt, np.array([int(g["seqlen"][0])], np.int32), dv, g["scale"][0], False)
    assert abs(lse[0, 0, 0] - g["lse"][0]) < 1e-13, "two-key LSE differs from the closed form"
    assert np.allclose(o[0, 0, 0], g["o"], rtol=0, atol=1e-13), "two-key O differs from the closed form"


def pin_score_shift(decode, seed=15):
    rng = np.random.default_rng(seed)
    d, dv, page = 576, 512, 64
    seqlens = [90, 33]
    r = rand_bits(rng, (d - dv,))
    rows = []
    for T in seqlens:
        x = rand_bits(rng, (T, 1, d))
        x[:, 0, dv:] = r                       # every key carries the same RoPE part
        rows.append(x)
    kc, bt = page_out(rows, page, rng)
    q1 = rand_bits(rng, (2, 1, 4, d))
    q2 = q1.copy()
    q2[..., dv:] = rand_bits(rng, (2, 1, 4, d - dv))
    sl = np.array(seqlens, np.int32)
    scale = 1 / 24
    o1, l1 = decode(q1, kc, bt, sl, dv, scale, False)
    o2, l2 = decode(q2, kc, bt, sl, dv, scale, False)
    rf = f64_of(r)
    shift = scale * ((f64_of(q2)[..., dv:] - f64_of(q1)[..., dv:]) @ rf)
    assert np.allclose(l2 - l1, shift, rtol=0, atol=1e-11), "LSE does not shift with the RoPE score offset"
    assert np.allclose(o1, o2, rtol=1e-11, atol=1e-12), "O changed under a common score shift"


def pin_causal_consistency(decode, seed=16):
    rng = np.random.default_rng(seed)
    d, dv, page, s_q = 576, 512, 64, 4
    seqlens = [70, 130]
    q = rand_bits(rng, (2, s_q, 4, d))
    rows = [rand_bits(rng, (T, 1, d)) for T in seqlens]
    kc, bt = page_out(rows, page, rng)
    o, lse = decode(q, kc, bt, np.array(seqlens, np.int32), dv, 1 / 24, True)
    for i in range(s_q):
        sl_i = np.array([T - s_q + i + 1 for T in seqlens], np.int32)
        o1, l1 = decode(np.ascontiguousarray(q[:, i:i + 1]), kc, bt, sl_i, dv, 1 / 24, False)
        assert np.allclose(o[:, i], o1[:, 0], rtol=1e-12, atol=1e-14), "causal query differs from its prefix call"
        assert np.allclose(lse[:, i], l1[:, 0], rtol=0, atol=1e-12), "causal LSE differs from its prefix call"


def pin_zero_visible(decode, seed=17):
    rng = np.random.default_rng(seed)
    d, dv = 576, 512
    q = rand_bits(rng, (2, 3, 2, d))
    rows = [rand_bits(rng, (0, 1, d)), rand_bits(rng, (2, 1, d))]
    kc, bt = page_out(rows, 64, rng)
    o, lse = decode(q, kc, bt, np.array([0, 2], np.int32), dv, 1 / 24, True)
    assert np.all(lse[0] == -math.inf) and np.all(o[0] == 0), "empty sequence must give O=0, LSE=-inf"
    assert np.all(lse[1, 0] == -math.inf) and np.all(o[1, 0] == 0), "causal row with no key must be empty"
    assert np.all(np.isfinite(lse[1, 1:])), "rows with visible keys must have finite LSE"


def pin_kv_head_groups(decode, seed=18):
    rng = np.random.default_rng(seed)
    d, dv, h_q, h_kv = 576, 512, 8, 2
    seqlens = [77, 5]
    q = rand_bits(rng, (2, 1, h_q, d))
    rows = [rand_bits(rng, (T, h_kv, d)) for T in seqlens]
    kc, bt = page_out(rows, 64, rng)
    sl = np.array(seqlens, np.int32)
    o, lse = decode(q, kc, bt, sl, dv, 1 / 24, False)
    per = h_q // h_kv
    for g in range(h_kv):
        kg = np.ascontiguousarray(kc[:, :, g:g + 1])
        qg = np.ascontiguousarray(q[:, :, g * per:(g + 1) * per])
        og, lg = decode(qg, kg, bt, sl, dv, 1 / 24, False)
        assert np.array_equal(o[:, :, g * per:(g + 1) * per], og), "head group reads the wrong KV head"
        assert np.array_equal(lse[:, :, g * per:(g + 1) * per], lg)


def pin_sampled_rows(decode, seed=19):
    rng = np.random.default_rng(seed)
    d, dv = 576, 512
    seqlens = [100, 250]
    q = rand_bits(rng, (2, 2, 4, d))
    rows = [rand_bits(rng, (T, 1, d)) for T in seqlens]
    kc, bt = page_out(rows, 64, rng)
    sl = np.array(seqlens, np.int32)
    o, lse = decode(q, kc, bt, sl, dv, 1 / 24, True)
    pick = np.array([0, 5, 9, 15], np.int64)
    os_, ls_ = decode(q, kc, bt, sl, dv, 1 / 24, True, rows=pick)
    assert np.array_equal(os_, o.reshape(-1, dv)[pick]) and np.array_equal(ls_, lse.reshape(-1)[pick])


def pin_saturated_softmax(decode, seed=20):
    rng = np.random.default_rng(seed)
    d, dv, T, win = 576, 512, 70, 41
    x = rand_bits(rng, (T, 1, d), scale=0.01)
    x[win, 0, :] = bf16_bits_of(np.full(d, 2.0))      # the winning key
    q = bf16_bits_of(np.full((1, 1, 1, d), 1.0))
    kc, bt = page_out([x], 64, rng)
    scale = 1.0                                        # s_win = 2 * 576 = 1152
    o, lse = decode(q, kc, bt, np.array([T], np.int32), dv, scale, False)
    s_win = 2.0 * d
    assert abs(lse[0, 0, 0] - s_win) < 1e-9, "saturated LSE must equal the top score"
    assert np.allclose(o[0, 0, 0], 2.0, rtol=0, atol=1e-12), "saturated O must equal the top key's V row"


ALL_PINS = [pin_brute_force, pin_permutation, pin_q_zero, pin_seqlen_one, pin_two_key_golden,
            pin_score_shift, pin_causal_consistency, pin_zero_visible, pin_kv_head_groups,
            pin_sampled_rows, pin_saturated_softmax]


# ---------------------------------------------------------------- e4m3 cache pins
E4M3_NAN_CODES = (0x7F, 0xFF)


def e4m3_codes_of(x) -> np.ndarray:
    """Round values to e4m3 codes (torch's cast, nearest even) after clamping to +-448."""
    t = torch.as_tensor(np.asarray(x, dtype=np.float32)).clamp(-448.0, 448.0).to(torch.float8_e4m3fn)
    return t.view(torch.uint8).numpy().copy()


def e4m3_values_of(codes) -> np.ndarray:
    """fp64 values of e4m3 codes through torch's own decoding."""
    return torch.from_numpy(np.ascontiguousarray(codes, dtype=np.uint8)).view(torch.float8_e4m3fn).to(
        torch.float64).numpy()


def fp8_pages(codes, scales) -> np.ndarray:
    """Pack codes uint8 [n, page, d] and scales fp32 [n, page] into [n, page * d + page * 4]."""
    n, page, d = codes.shape
    out = np.empty((n, page * d + page * 4), dtype=np.uint8)
    out[:, :page * d] = codes.reshape(n, page * d)
    out[:, page * d:] = np.ascontiguousarray(scales, dtype="<f4").view(np.uint8).reshape(n, page * 4)
    return out


def _fp8_case(rng, seqlens, d, page, pow2_scales):
    """Random e4m3 cache for `seqlens`: (pages, dequantized fp64 [pool, page, d], block_table).

    Rows past each sequence's end and unused pages hold random codes (NaN codes
    included) and NaN scales: no decode may read them."""
    n_pages = [(T + page - 1) // page for T in seqlens]
    pool = sum(n_pages) + 2
    codes = e4m3_codes_of(rng.standard_normal((pool, page, d)) * 8.0)
    if pow2_scales:
        scales = np.exp2(rng.integers(-5, 0, size=(pool, page))).astype(np.float32)
    else:
        scales = rng.uniform(0.01, 0.2, size=(pool, page)).astype(np.float32)
    used = np.zeros((pool, page), dtype=bool)
    perm = rng.permutation(pool).astype(np.int32)
    bt = np.zeros((len(seqlens), max(n_pages)), dtype=np.int32)
    cur = 0
    for b, T in enumerate(seqlens):
        for p in range(n_pages[b]):
            bt[b, p] = perm[cur]
            used[perm[cur], :min(page, T - p * page)] = True
            cur += 1
    junk = rng.integers(0, 256, size=codes.shape).astype(np.uint8)
    junk[..., :2] = E4M3_NAN_CODES
    codes = np.where(used[..., None], codes, junk)
    scales = np.where(used, scales, np.float32(np.nan)).astype(np.float32)
    deq = e4m3_values_of(codes) * scales[..., None].astype(np.float64)
    return fp8_pages(codes, scales), deq, used, bt


def pin_e4m3_codes(decode, decode_fp8, e4m3):
    codes = np.arange(256, dtype=np.uint8)
    v = e4m3(codes)
    t = e4m3_values_of(codes)
    assert np.array_equal(np.isnan(v), np.isnan(t)), "NaN codes differ from torch's e4m3"
    assert np.array_equal(v[~np.isnan(v)], t[~np.isnan(t)]), "e4m3 values differ from torch's"
    assert v[0x38] == 1.0 and v[0x7E] == 448.0 and v[0xFE] == -448.0, "e4m3 normal landmarks"
    assert v[0x01] == 2.0 ** -9 and v[0x07] == 7 * 2.0 ** -9 and v[0x08] == 2.0 ** -6, "e4m3 subnormal landmarks"
    assert np.isnan(v).sum() == 2 and all(np.isnan(v[c]) for c in E4M3_NAN_CODES), "e4m3 has exactly two NaNs"
    assert v[0x80] == 0.0 and math.copysign(1.0, v[0x80]) == -1.0, "0x80 is -0"


def pin_fp8_matches_bf16(decode, decode_fp8, e4m3, seed=21):
    rng = np.random.default_rng(seed)
    d, dv, page = 576, 512, 64
    for seqlens, s_q, h_q, causal in (([130, 64, 7], 2, 8, True), ([1, 200], 1, 16, False)):
        pages, deq, used, bt = _fp8_case(rng, seqlens, d, page, pow2_scales=True)
        # the same rows as a bf16 cache: every dequantized value is a bf16 value
        kc = bf16_bits_of(np.where(used[..., None], deq, 1e4 * rng.standard_normal(deq.shape)))[:, :, None, :]
        assert np.array_equal(f64_of(kc[:, :, 0, :])[used], deq[used]), "dequantized rows must be bf16-exact"
        q = rand_bits(rng, (len(seqlens), s_q, h_q, d))
        sl = np.array(seqlens, np.int32)
        o8, l8 = decode_fp8(q, pages, bt, sl, dv, 1.0 / 24, causal)
        o, l = decode(q, kc, bt, sl, dv, 1.0 / 24, causal)
        assert np.array_equal(l8, l), "e4m3 LSE differs from the bf16 decode of the same rows"
        assert np.array_equal(o8, o), "e4m3 O differs from the bf16 decode of the same rows"


def pin_fp8_scale_linearity(decode, decode_fp8, e4m3, seed=22):
    rng = np.random.default_rng(seed)
    d, dv, page = 576, 512, 64
    seqlens = [100, 65]
    pages, deq, used, bt = _fp8_case(rng, seqlens, d, page, pow2_scales=False)
    q = rand_bits(rng, (2, 1, 16, d))
    sl = np.array(seqlens, np.int32)
    o1, l1 = decode_fp8(q, pages, bt, sl, dv, 1.0 / 24, False)
    doubled = pages.copy()
    sc = doubled[:, page * d:].view("<f4")
    sc *= 2.0
    q_half = bf16_bits_of(f64_of(q) / 2.0)
    o2, l2 = decode_fp8(q_half, doubled, bt, sl, dv, 1.0 / 24, False)
    assert np.array_equal(l2, l1), "scores must not change when q halves and the scales double"
    assert np.array_equal(o2, 2.0 * o1), "O must double with the scales"


FP8_PINS = [pin_e4m3_codes, pin_fp8_matches_bf16, pin_fp8_scale_linearity]



# ---------------------------------------------------------------- sparse top-k pins
def _sparse_brute(q_bits, rows_per_seq, seqlens, indices, dv, scale, h_kv):
    qf = f64_of(q_bits)
    b, s_q, h_q, d = qf.shape
    o = np.zeros((b, s_q, h_q, dv))
    lse = np.zeros((b, s_q, h_q))
    for bi in range(b):
        kf = f64_of(rows_per_seq[bi])                      # [T, h_kv, d]
        for i in range(s_q):
            sel = [int(j) for j in indices[bi, i] if 0 <= j < seqlens[bi]]
            for h in range(h_q):
                g = h // (h_q // h_kv)
                if not sel:
                    lse[bi, i, h] = -math.inf
                    continue
                K = kf[sel, g, :]                          # repeats kept
                e = np.exp(scale * (K @ qf[bi, i, h]))
                o[bi, i, h] = (e @ K[:, :dv]) / e.sum()
                lse[bi, i, h] = math.log(e.sum())
    return o, lse


def _random_lists(rng, seqlens, s_q, topk):
    """Lists mixing valid positions, repeats, -1 padding and positions >= T."""
    lists = np.full((len(seqlens), s_q, topk), -1, np.int32)
    for b, T in enumerate(seqlens):
        for i in range(s_q):
            n = int(rng.integers(0, topk + 1))
            vals = rng.integers(-1, T + 2, size=n) if T > 0 else rng.integers(-1, 3, size=n)
            lists[b, i, :n] = vals
            if T > 0 and n >= 2:
                lists[b, i, 1] = lists[b, i, 0] if lists[b, i, 0] >= 0 else T - 1   # a repeat
            if n >= 3:
                lists[b, i, 2] = T                                               # one past the end
    return lists


def pin_sparse_brute_force(decode, decode_sparse, seed=31):
    rng = np.random.default_rng(seed)
    cases = [
        # (b, s_q, h_q, h_kv, seqlens, topk, d, dv, page)
        (2, 1, 16, 1, [100, 37], 48, 576, 512, 64),
        (3, 2, 4, 1, [1, 200, 0], 70, 576, 512, 64),
        (2, 3, 8, 2, [130, 65], 33, 512, 512, 64),
        (1, 4, 2, 1, [9], 12, 40, 24, 4),
    ]
    for (b, s_q, h_q, h_kv, seqlens, topk, d, dv, page) in cases:
        q = rand_bits(rng, (b, s_q, h_q, d))
        rows = [rand_bits(rng, (max(T, 1), h_kv, d)) for T in seqlens]
        kc, bt = page_out(rows, page, rng)
        idx = _random_lists(rng, seqlens, s_q, topk)
        scale = 1.0 / math.sqrt(d)
        sl = np.array(seqlens, np.int32)
        o, lse = decode_sparse(q, kc, bt, sl, idx, dv, scale)
        o_ref, lse_ref = _sparse_brute(q, rows, seqlens, idx, dv, scale, h_kv)
        assert np.array_equal(np.isneginf(lse), np.isneginf(lse_ref)), "rows without valid entries differ"
        fin = ~np.isneginf(lse_ref)
        assert np.allclose(lse[fin], lse_ref[fin], rtol=0, atol=1e-11), "sparse LSE differs from brute force"
        assert np.allclose(o, o_ref, rtol=1e-11, atol=1e-12), "sparse O differs from brute force"


def pin_sparse_full_list(decode, decode_sparse, seed=32):
    rng = np.random.default_rng(seed)
    d, dv, page = 576, 512, 64
    seqlens = [150, 64, 1]
    q = rand_bits(rng, (3, 1, 8, d))
    kc, bt = page_out([rand_bits(rng, (T, 1, d)) for T in seqlens], page, rng)
    sl = np.array(seqlens, np.int32)
    idx = np.full((3, 1, 160), -1, np.int32)
    for b, T in enumerate(seqlens):
        idx[b, 0, :T] = np.arange(T)
    o, lse = decode_sparse(q, kc, bt, sl, idx, dv, 1.0 / 24)
    o_d, lse_d = decode(q, kc, bt, sl, dv, 1.0 / 24, False)
    assert np.array_equal(lse, lse_d) and np.array_equal(o, o_d), "the full list must give the dense decode"


def pin_sparse_order(decode, decode_sparse, seed=33):
    rng = np.random.default_rng(seed)
    d, dv, page = 576, 512, 64
    seqlens = [300, 90]
    q = rand_bits(rng, (2, 2, 4, d))
    kc, bt = page_out([rand_bits(rng, (T, 1, d)) for T in seqlens], page, rng)
    sl = np.array(seqlens, np.int32)
    idx = np.stack([np.stack([rng.choice(T, size=40, replace=False) for _ in range(2)]) for T in seqlens]).astype(
        np.int32)
    o, lse = decode_sparse(q, kc, bt, sl, idx, dv, 1.0 / 24)
    perm = idx[:, :, rng.permutation(40)]
    o_p, lse_p = decode_sparse(q, kc, bt, sl, perm, dv, 1.0 / 24)
    assert np.allclose(lse_p, lse, rtol=0, atol=1e-12) and np.allclose(o_p, o, rtol=1e-12, atol=1e-14), \
        "the order of a list must not matter"
    padded = np.concatenate([idx, np.full((2, 2, 3), -1, np.int32), np.stack([sl, sl], axis=1)[:, :, None]], axis=2)
    o_x, lse_x = decode_sparse(q, kc, bt, sl, padded, dv, 1.0 / 24)
    assert np.array_equal(lse_x, lse) and np.array_equal(o_x, o), "ignored entries must change nothing"


SPARSE_PINS = [pin_sparse_brute_force, pin_sparse_full_list, pin_sparse_order]
