"""Pins of the CPU oracle against what the curta-core page ("The inference core") and
mathematics fix: printed values, closed forms, textbook routines, brute force on tiny
inputs and real-valued error bounds.  Each test names the step it pins; a plausible
mistake in the oracle (a dropped term, a wrong shift or sign, a floor instead of a
truncation, a transposed operand) fails at least one of them."""
import json
import math
import os

import numpy as np
import pytest

import oracle
import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "page_facts.json")
M64 = 2**64


def facts():
    with open(GOLDEN) as f:
        return json.load(f)


def s64(v: int) -> int:
    v %= M64
    return v - M64 if v >= 2**63 else v


# ---------------------------------------------------------------- isqrt (textbook)

def test_isqrt_matches_math_isqrt():
    vals = list(range(0, 70000)) + [42950, 4295010246, M64 - 1, 2**63, 2**62]
    rng = np.random.default_rng(1)
    for k in list(rng.integers(1, 2**32 - 1, 3000, dtype=np.uint64)) + [2**32 - 1, 65536, 207, 208]:
        k = int(k)
        vals += [k * k - 1, k * k, k * k + 1, min(k * k + 2 * k, M64 - 1)]
    for v in vals:
        assert oracle.isqrt(v) == math.isqrt(v), v


def test_isqrt_epsilon_floor():
    # an all-zero vector normalises with rms = isqrt(42,950) = 207 (207^2 <= 42950 < 208^2)
    assert oracle.isqrt(facts()["rms_epsilon"]["value"]) == 207


# ---------------------------------------------------------------- embedding (closed form)

def test_embed_is_floor_of_dequantised_row():
    row = np.arange(256, dtype=np.uint8)
    for scale in (0, 1, 255, 2**21 + 12345, 2**32 - 1):
        got = oracle.embed(row, scale)
        want = [((b - 128) * scale) // 256 for b in range(256)]   # Python // floors
        assert got.tolist() == want


# ---------------------------------------------------------------- RMS normalization

def test_rmsnorm_zero_vector():
    assert oracle.rmsnorm(np.zeros(64, np.int64), np.full(64, 2**24, np.int32)).tolist() == [0] * 64


def test_rmsnorm_unit_vector_unit_weight_is_exact():
    # x = 1.0 everywhere, w = 1.0: mean square 2^32, rms = isqrt(2^32 + 42950) = 65536, y = 1.0
    y = oracle.rmsnorm(np.full(4096, 2**16, np.int64), np.full(4096, 2**24, np.int32))
    assert (y == 2**16).all()


def test_rmsnorm_division_truncates_then_shift_floors():
    # one element x = 1: rms = isqrt(1 + 42950) = 207.  x*w = -(256*207 + 1):
    # truncating division gives -256 and >> 8 gives -1; a floor division would give -257, -2.
    assert oracle.isqrt(1 + 42950) == 207
    assert oracle.rmsnorm(np.array([1]), np.array([-(256 * 207 + 1)])).tolist() == [-1]
    assert oracle.rmsnorm(np.array([1]), np.array([256 * 207 + 1])).tolist() == [1]
    # x*w = -(207*255): the quotient -255 is exact and the arithmetic shift floors to -1
    assert oracle.rmsnorm(np.array([1]), np.array([-207 * 255])).tolist() == [-1]
    assert oracle.rmsnorm(np.array([1]), np.array([-207 * 256])).tolist() == [-1]
    assert oracle.rmsnorm(np.array([1]), np.array([-207 * 257])).tolist() == [-2]


def test_rmsnorm_within_fixed_point_bound_of_real_rmsnorm():
    rng = np.random.default_rng(7)
    for n in (1, 7, 64, 4096):
        for scale in (0.01, 1.0, 30.0):
            xf = rng.normal(0, scale, n)
            wf = rng.uniform(0.5, 1.5, n)
            x = np.round(xf * 2**16).astype(np.int64)
            w = np.round(wf * 2**24).astype(np.int32)
            y = oracle.rmsnorm(x, w)
            xr = x / 2**16
            rms = math.sqrt(float(np.mean(xr * xr)) + 1e-5)
            want = xr * (w / 2**24) / rms * 2**16        # real RMSNorm in units of 2^-16
            rms_fixed = math.sqrt(float(np.mean(xr * xr)) * 2**32 + 42950)
            bound = np.abs(want) * (1.0 / max(rms_fixed - 1, 1)) + 2.5
            assert (np.abs(y - want) <= bound).all(), (n, scale)


# ---------------------------------------------------------------- matrix row

def _matrow_signed(W, s, x):
    """The signed dot product the page says the +128 form equals, wrapped to 64 bits."""
    out = []
    for r in range(W.shape[0]):
        acc = sum((int(W[r, c]) - 128) * int(x[c]) for c in range(W.shape[1]))
        out.append(s64(s64(acc) * int(s[r])) >> 24)
    return out


def test_matrow_equals_signed_dot_product_brute_force():
    rng = np.random.default_rng(3)
    extremes = [0, 1, -1, 2**62, -2**62, 2**63 - 1, -2**63, 2**31, -2**31 - 7]
    for cols in list(range(1, 41)) + [64, 172]:
        rows = 3
        W = rng.integers(0, 256, (rows, cols), dtype=np.uint8)
        W[0, :] = 0
        W[1, : cols // 2] = 255
        x = rng.integers(-2**40, 2**40, cols, dtype=np.int64)
        x[: min(cols, len(extremes))] = extremes[: min(cols, len(extremes))]
        s = np.array([1, 2**24, 2**32 - 1], dtype=np.uint32)
        assert oracle.matrow(W, s, x).tolist() == _matrow_signed(W, s, x), cols


def test_matrow_without_wrap_is_exact_floor():
    rng = np.random.default_rng(4)
    W = rng.integers(0, 256, (16, 300), dtype=np.uint8)
    x = rng.integers(-8 * 2**16, 8 * 2**16, 300, dtype=np.int64)
    s = rng.integers(2**20, 2**24, 16, dtype=np.uint32)
    want = [(sum((int(W[r, c]) - 128) * int(x[c]) for c in range(300)) * int(s[r])) // 2**24
            for r in range(16)]
    assert oracle.matrow(W, s, x).tolist() == want


def test_matrow_identity_row():
    # weight 1 (byte 129) on the diagonal, scale 1.0: y = x
    n = 37
    W = np.full((n, n), 128, np.uint8)
    np.fill_diagonal(W, 129)
    x = np.arange(-18, 19, dtype=np.int64) * 123457
    assert oracle.matrow(W, np.full(n, 2**24, np.uint32), x).tolist() == x.tolist()


def test_matrow_pitch_and_cols():
    rng = np.random.default_rng(5)
    W = rng.integers(0, 256, (5, 48), dtype=np.uint8)
    x = rng.integers(-2**20, 2**20, 48, dtype=np.int64)
    s = rng.integers(2**20, 2**24, 5, dtype=np.uint32)
    full = oracle.matrow(W[:, :45].copy(), s, x[:45])
    assert oracle.matrow(W, s, x, cols=45).tolist() == full.tolist()


# ---------------------------------------------------------------- cache fit check

def test_fits32_boundaries():
    c = facts()["cache_word_bits"]
    assert oracle.fits32(c["max"]) and oracle.fits32(c["min"]) and oracle.fits32(0)
    assert not oracle.fits32(c["max"] + 1) and not oracle.fits32(c["min"] - 1)
    assert not oracle.fits32(2**63 - 1) and not oracle.fits32(-2**63)


# ---------------------------------------------------------------- rotary

def test_rotary_position_zero_is_identity():
    tab = synth.rope_table(4, 16)
    assert (tab[0, :, 0] == 2**24).all() and (tab[0, :, 1] == 0).all()
    for a, b in ((5, -7), (2**38, -2**38), (-1, 1), (2**31 - 1, -2**31)):
        assert oracle.rotate(a, b, 2**24, 0) == (a, b)
    # reading r7: the products wrap in 64 bits, so 2^40 * 2^24 = 2^64 wraps to zero
    assert oracle.rotate(2**40, 0, 2**24, 0) == (0, 0)


def test_rotary_quarter_turn_and_real_rotation():
    # cos = 0, sin = 1: (a, b) -> (-b, a)
    assert oracle.rotate(3 * 2**16, 5 * 2**16, 0, 2**24) == (-5 * 2**16, 3 * 2**16)
    rng = np.random.default_rng(9)
    for _ in range(500):
        a, b = (int(v) for v in rng.integers(-2**31, 2**31, 2))
        th = float(rng.uniform(-math.pi, math.pi))
        c, s = round(math.cos(th) * 2**24), round(math.sin(th) * 2**24)
        a2, b2 = oracle.rotate(a, b, c, s)
        assert a2 == (a * c - b * s) >> 24 and b2 == (a * s + b * c) >> 24
        # and within rounding of the real rotation
        assert abs(a2 - (a * math.cos(th) - b * math.sin(th))) <= 1 + (abs(a) + abs(b)) * 2**-23
        assert abs(b2 - (a * math.sin(th) + b * math.cos(th))) <= 1 + (abs(a) + abs(b)) * 2**-23


# ---------------------------------------------------------------- attention

EXP = synth.exp_table()


def test_exp_table_page_facts():
    f = facts()["exp_table"]
    assert EXP.size == f["entries"] and int(EXP[0]) == f["entry0"] == 2**30
    for i in (1, 256, 2048, 4096):
        assert abs(int(EXP[i]) - math.exp(-i / 256) * 2**30) <= 0.5


def test_attention_single_position_returns_value():
    rng = np.random.default_rng(11)
    for hd in (8, 16, 64, 128):
        q = rng.integers(-2**20, 2**20, hd, dtype=np.int64)
        K = rng.integers(-2**20, 2**20, (1, hd), dtype=np.int32)
        V = rng.integers(-2**31, 2**31, (1, hd), dtype=np.int64).astype(np.int32)
        out, probs = oracle.attention_head(q, K, V, synth.inv_sqrt_head(hd), EXP)
        assert probs.tolist() == [2**24]
        assert out.tolist() == V[0].astype(np.int64).tolist()


def test_attention_equal_scores_closed_form():
    rng = np.random.default_rng(12)
    for p in (1, 2, 3, 7, 100):
        hd = 16
        q = rng.integers(-2**18, 2**18, hd, dtype=np.int64)
        k = rng.integers(-2**18, 2**18, hd, dtype=np.int32)
        K = np.tile(k, (p, 1))
        V = rng.integers(-2**30, 2**30, (p, hd), dtype=np.int32)
        out, probs = oracle.attention_head(q, K, V, 2**22, EXP)
        P = 2**24 // p
        assert probs.tolist() == [P] * p
        assert out.tolist() == [(P * int(V[:, j].astype(np.int64).sum())) >> 24 for j in range(hd)]


def test_attention_exp_index_and_cap():
    # q = (1.0, 0), inv = 1.0: the score of position t is its first key element.
    # Differences from the largest: 0, 2^20 - 1 (index 4095), 2^20 (4096), 2^21 (capped 4096), 255 (0)
    q = np.array([2**16, 0], np.int64)
    top = 2**21
    ks = [top, top - (2**20 - 1), top - 2**20, 0, top - 255]
    K = np.array([[k, 0] for k in ks], np.int32)
    V = np.zeros((5, 2), np.int32)
    _, probs = oracle.attention_head(q, K, V, 2**24, EXP)
    idx = [0, 4095, 4096, 4096, 0]
    Z = sum(int(EXP[i]) for i in idx)
    assert probs.tolist() == [(int(EXP[i]) << 24) // Z for i in idx]


def test_attention_near_real_softmax():
    rng = np.random.default_rng(13)
    for p, hd in ((5, 8), (40, 16), (300, 64)):
        qf = rng.normal(0, 1, hd)
        kf = rng.normal(0, 1, (p, hd))
        vf = rng.normal(0, 1, (p, hd))
        q = np.round(qf * 2**16).astype(np.int64)
        K = np.round(kf * 2**16).astype(np.int32)
        V = np.round(vf * 2**16).astype(np.int32)
        inv = synth.inv_sqrt_head(hd)
        out, probs = oracle.attention_head(q, K, V, inv, EXP)
        sc = (K / 2**16) @ (q / 2**16) / math.sqrt(hd)
        e = np.exp(sc - sc.max())
        pr = e / e.sum()
        # the table quantises score differences to 1/256 (relative error <= e^(1/256) - 1)
        assert np.abs(probs / 2**24 - pr).max() <= 0.01
        want = pr @ (V / 2**16)
        assert np.abs(out / 2**16 - want).max() <= 0.02


# ---------------------------------------------------------------- SiLU

SILU = synth.silu_table()


def test_silu_edges():
    f = facts()["silu_table"]
    up, lo = f["upper"], f["lower"]
    assert up == 16 * 2**16 and lo == -16 * 2**16
    assert oracle.silu(up, SILU) == up and oracle.silu(up + 12345, SILU) == up + 12345
    assert oracle.silu(up - 1, SILU) == int(SILU[4095])
    assert oracle.silu(lo, SILU) == 0 and oracle.silu(lo - 5, SILU) == 0
    assert oracle.silu(lo + 1, SILU) == int(SILU[0])
    assert oracle.silu(0, SILU) == int(SILU[2048]) == 0
    assert oracle.silu(-1, SILU) == int(SILU[2047])           # (2^20 - 1) >> 9 = 2047
    assert oracle.silu(511, SILU) == int(SILU[2048]) and oracle.silu(512, SILU) == int(SILU[2049])


def test_silu_near_real_function():
    rng = np.random.default_rng(14)
    for g in rng.integers(-17 * 2**16, 17 * 2**16, 4000):
        g = int(g)
        x = g / 2**16
        real = x / (1 + math.exp(-x)) * 2**16 if x > -700 else 0.0
        # one table step of 1/128 at slope at most 1.1, plus rounding
        assert abs(oracle.silu(g, SILU) - real) <= 1.1 * 2**16 / 128 + 1


def test_silu_gate_closed_form():
    g = np.array([2**20, 2**21, -2**20, 0, 3 * 2**20], np.int64)
    u = np.array([3 * 2**16, -5, 7, 9, -(2**16) - 1], np.int64)
    h = oracle.silu_gate(g, u, SILU)
    want = [(int(oracle.silu(int(a), SILU)) * int(b)) >> 16 for a, b in zip(g, u)]
    assert h.tolist() == want
    assert h[0] == 3 * 2**20 and h[2] == 0 and h[3] == 0


# ---------------------------------------------------------------- maximum pass

def test_argmax_first_of_ties():
    assert oracle.argmax(np.array([3, 9, 9, 1])) == 1
    assert oracle.argmax(np.array([-5, -5, -5])) == 0
    assert oracle.argmax(np.array([-2**63, 2**63 - 1])) == 1
    rng = np.random.default_rng(15)
    for _ in range(50):
        v = rng.integers(-3, 3, 64)
        assert oracle.argmax(v) == int(np.argmax(v))         # numpy also returns the first


# ---------------------------------------------------------------- state sizes printed on the page

def test_page_state_sizes():
    f = facts()["state_sizes"]
    for c in f["cases"]:
        got = oracle.page_state_size(c["config"], c["prompt_bytes"], c["max_tokens"])
        assert got + f["account_header_bytes"] == c["account_bytes"], c


def test_xorshift64star_generator():
    f = facts()["xorshift64star"]
    mult, zero = int(f["multiplier"], 16), int(f["zero_seed_state"], 16)

    def step(x):
        x ^= x >> 12
        x ^= (x << 25) % M64
        x ^= x >> 27
        return x, (x * mult) % M64

    x, want = zero, []
    for _ in range(5):
        x, o = step(x)
        want.append(o)
    assert synth.xs64s_sequence(0, 5) == want


# ---------------------------------------------------------------- sampling (phase 19 above zero)

def _gf2_apply(cols, v):
    """The GF(2) matrix with the given column images applied to the 64-bit vector v."""
    out = 0
    j = 0
    while v:
        if v & 1:
            out ^= cols[j]
        v >>= 1
        j += 1
    return out


def _gf2_mul(a, b):
    return [_gf2_apply(a, c) for c in b]


def _gf2_pow(a, e):
    r = [1 << j for j in range(64)]
    while e:
        if e & 1:
            r = _gf2_mul(r, a)
        a = _gf2_mul(a, a)
        e >>= 1
    return r


def test_sampling_generator_has_the_full_xorshift_period():
    """The oracle's state step is linear over GF(2) and its matrix has order exactly
    2^64 - 1, the maximal period Marsaglia's xorshift theorem gives for the triple
    (12, 25, 27): a wrong shift amount or direction breaks it.  Its output is the state
    times the page's multiplier, and the zero seed's sequence matches the input generator's
    (itself pinned to the page above)."""
    f = facts()["xorshift64star"]
    mult, zero = int(f["multiplier"], 16), int(f["zero_seed_state"], 16)
    step = lambda x: oracle.xorshift_next(x)[0]
    cols = [step(1 << j) for j in range(64)]
    rng = np.random.default_rng(3)
    for _ in range(20):
        a, b = (int(v) for v in rng.integers(0, 2**63, 2, dtype=np.uint64))
        assert step(a ^ b) == step(a) ^ step(b)
        assert step(a) == _gf2_apply(cols, a)
    order = 2**64 - 1
    ident = [1 << j for j in range(64)]
    assert _gf2_pow(cols, order) == ident
    for p in (3, 5, 17, 257, 641, 65537, 6700417):            # the primes of 2^64 - 1
        assert order % p == 0
        assert _gf2_pow(cols, order // p) != ident
    x, outs = zero, []
    for _ in range(6):
        x, o = oracle.xorshift_next(x)
        assert o == (x * mult) % M64
        outs.append(o)
    assert outs == synth.xs64s_sequence(0, 6)


def test_sample_index_is_the_table_rule_at_temperature_one():
    """At temperature 1 (1 << 16) the index is the exponential table's own rule, d >> 8
    capped at 4096; temperature 2 halves the step and 1/2 doubles it; huge differences cap
    without wrapping."""
    rng = np.random.default_rng(4)
    for _ in range(300):
        m = int(rng.integers(-2**40, 2**40))
        d = int(rng.integers(0, 2**22))
        assert oracle.sample_index(m, m - d, 1 << 16) == min(d >> 8, 4096)
        assert oracle.sample_index(m, m - d, 1 << 17) == min(d >> 9, 4096)
        assert oracle.sample_index(m, m - d, 1 << 15) == min(d >> 7, 4096)
    assert oracle.sample_index(2**63 - 1, -2**63, 1) == 4096
    assert oracle.sample_index(2**63 - 1, -2**63, 16 << 16) == 4096
    assert oracle.sample_index(5, 5, 1) == 0


def test_sample_index_is_exp_of_difference_over_temperature():
    """Real-valued check: the entry read is e^-(dl / T) to within one table step (1/256 in
    the exponent) plus the entry's rounding, for temperatures that are not powers of two."""
    tab = synth.exp_table()
    rng = np.random.default_rng(5)
    for _ in range(400):
        t = int(rng.integers(1, 16 << 16))
        d = int(rng.integers(0, 17 * t))
        idx = oracle.sample_index(0, -d, t)
        x = (d / 65536) / (t / 65536)
        if x >= 4097 / 256:
            assert idx == 4096
            continue
        assert idx == int(x * 256) or abs(x * 256 - round(x * 256)) < 1e-9
        got = tab[idx] / 2**30
        assert math.exp(-x) <= got * math.exp(1 / 256) + 1e-9
        assert got <= math.exp(-x) * math.exp(1 / 256) + 1e-9


def test_draw_walk_takes_the_first_entry_the_remainder_falls_inside():
    e = np.array([5, 0, 3, 7], dtype=np.uint64)
    want = {0: 0, 4: 0, 5: 2, 7: 2, 8: 3, 14: 3, 15: 4}
    for r, i in want.items():
        assert oracle.draw_walk(e, r) == i, r


def test_sample_temperature_zero_is_the_maximum_pass():
    v = np.array([3, 9, 9, 1], dtype=np.int64)
    r = oracle.sample(v, 0, synth.exp_table(), 77)
    assert r == {"token": 1, "state": 77, "max": 9, "sum": 0, "draw": 0}


def test_sample_equal_logits_closed_form():
    """Equal logits: every exponential is EXP[0] = 2^30, the sum is n * 2^30, and the draw
    picks entry draw // 2^30; the state advances exactly once."""
    tab = synth.exp_table()
    for n, t, seed in ((7, 1 << 16, 11), (1000, 3 << 16, 12345), (32000, 1, 2**63 + 9)):
        v = np.full(n, -42, dtype=np.int64)
        r = oracle.sample(v, t, tab, seed)
        out = synth.xs64s_sequence(seed, 1)[0]
        assert r["sum"] == n << 30
        assert r["draw"] == out % (n << 30)
        assert r["token"] == r["draw"] >> 30
        assert r["state"] == oracle.xorshift_next(seed)[0]
        assert r["max"] == -42


def test_sample_frequencies_follow_the_exponentials():
    """Many draws from one vector: each entry's frequency is its exponential over the sum
    (binomial 5-sigma bound).  Logits are spaced on the table's grid at temperature 1."""
    tab = synth.exp_table()
    ks = [0, 100, 256, 700, 4096, 5000]
    v = np.array([-256 * k for k in ks], dtype=np.int64)
    e = np.array([tab[min(k, 4096)] for k in ks], dtype=np.float64)
    p = e / e.sum()
    n = 20000
    counts = np.zeros(len(ks))
    state = 99
    for _ in range(n):
        r = oracle.sample(v, 1 << 16, tab, state)
        state = r["state"]
        counts[r["token"]] += 1
        assert r["sum"] == int(e.sum())
    for i in range(len(ks)):
        sd = math.sqrt(n * p[i] * (1 - p[i])) + 1
        assert abs(counts[i] - n * p[i]) <= 5 * sd, (i, counts[i], n * p[i])


# ---------------------------------------------------------------- tokenizer (phases 0 to 2)

def _blob(extra):
    """A vocabulary in the tokenizer file layout: the 3 specials, the 256 byte tokens, then
    `extra` (bytes, score) pairs."""
    import struct
    toks = [(b"<unk>", 0.0), (b"\n<s>\n", 0.0), (b"\n</s>\n", 0.0)]
    toks += [(("<0x%02X>" % i).encode(), 0.0) for i in range(256)] + list(extra)
    out = struct.pack("<I", max(len(t) for t, _ in toks))
    for t, sc in toks:
        out += struct.pack("<fi", sc, len(t)) + t
    return out, len(toks)


def _vocab(extra):
    blob, n = _blob(extra)
    v = oracle.Vocab(blob, n)
    ids = {t: i for i, (t, _) in enumerate(extra, start=259)}
    return v, ids


def test_encode_opening_token_and_space():
    """Phase 0: token 1, then the single-space token when the prompt has text."""
    v, ids = _vocab([(b" ", -1.0), (b"a", -1.0)])
    assert v.encode(b"") == (0, [1])
    assert v.encode(b"a") == (0, [1, ids[b" "], ids[b"a"]])
    v2, ids2 = _vocab([(b"a", -1.0)])                      # no space token: its byte token
    assert v2.encode(b"a") == (0, [1, 0x20 + 3, ids2[b"a"]])


def test_encode_byte_fallback():
    """Phase 1: a character with no token becomes one token per byte, id byte + 3."""
    v, ids = _vocab([(b" ", -1.0), (b"x", -1.0), ("é".encode(), -1.0)])
    rc, t = v.encode("x日é".encode())
    assert rc == 0
    assert t == [1, ids[b" "], ids[b"x"], 0xE6 + 3, 0x97 + 3, 0xA5 + 3, ids["é".encode()]]


def test_encode_merges_take_the_highest_score():
    """Phase 2: of all adjacent pairs whose joined text is a token, the best score merges
    first; merges repeat on the result."""
    v, ids = _vocab([(b" ", -1.0), (b"a", -1.0), (b"b", -1.0), (b"c", -1.0), (b"ab", -5.0), (b"bc", -1.0)])
    assert v.encode(b"abc") == (0, [1, ids[b" "], ids[b"a"], ids[b"bc"]])
    v, ids = _vocab([(b" ", -1.0), (b"a", -1.0), (b"b", -1.0), (b"c", -1.0), (b"ab", -1.0), (b"abc", -2.0)])
    assert v.encode(b"abc") == (0, [1, ids[b" "], ids[b"abc"]])
    v, ids = _vocab([(b" ", -1.0), (b"a", -1.0), (b"aa", -1.0), (b" a", -9.0)])
    # "aaa": the two (a, a) pairs tie, the leftmost merges (r24); then " a" is not
    # reachable because the space now precedes "aa"
    assert v.encode(b"aaa") == (0, [1, ids[b" "], ids[b"aa"], ids[b"a"]])


def test_encode_rejects_bad_prompts():
    v, _ = _vocab([(b" ", -1.0)])
    assert v.encode(b"a\x00b")[0] == 6                     # a zero byte
    assert v.encode(b"\xff")[0] == 6                       # not UTF-8
    assert v.encode(b"\xc3")[0] == 6                       # truncated character
    assert v.encode(b"\xc0\x80")[0] == 6                   # overlong
    assert v.encode(b"a" * 1025)[0] == 6                   # over 1,024 bytes
    assert v.encode(b"a" * 1024)[0] == 0


def test_token_text_rules():
    """Token text: the bytes, a leading space dropped right after the opening token, <0xXX>
    as one byte, nothing for tokens 1 and 2."""
    v, ids = _vocab([(b" hi", -1.0)])
    assert v.piece(1, ids[b" hi"]) == b"hi"
    assert v.piece(7, ids[b" hi"]) == b" hi"
    assert v.piece(5, 0x41 + 3) == b"A"
    assert v.piece(5, 1) == b"" and v.piece(5, 2) == b""
    assert v.decode([1, ids[b" hi"], ids[b" hi"], 2]) == b"hi hi"


def test_encode_fixed_point_and_round_trip_on_synthetic_vocabularies():
    """For seeded prompts: decoding the encoding gives the prompt back, and no adjacent pair
    of the result joins into a token (the merges ran to the end)."""
    for n, seed in ((512, 0x5EED0011), (32000, 0x5EED0003)):
        blob = synth.tokenizer_blob(n, seed)
        v = oracle.Vocab(blob, n)
        pieces = synth.vocab_pieces(blob)
        for run in range(6):
            text = synth.prompt_text(80, seed, run, blob)
            rc, ids = v.encode(text)
            assert rc == 0
            assert v.decode(ids) == text
            for a, b in zip(ids, ids[1:]):
                assert v.lookup(pieces[a] + pieces[b]) < 0
