"""The C-ABI library builds for sm_103a, loads, and exports every function include/ck.h
declares; host builds of its integer routines match their definitions.  No GPU needed."""
import ctypes
import math
import os
import re

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "ck.h")


@pytest.fixture(scope="module")
def ck():
    import fixed_point_int8_gb300 as ck
    from fixed_point_int8_gb300 import build
    build.build()
    return ck


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(ck_[a-z_0-9]+)\s*\(", text)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for want in ("ck_load_model", "ck_init_state", "ck_turn", "ck_logits", "ck_argmax", "ck_matrow"):
        assert want in names


def test_library_exports_every_declared_symbol(ck):
    lib = ctypes.CDLL(ck.build.LIB)
    missing = [n for n in declared_functions() if not hasattr(lib, n)]
    assert not missing, missing
    assert "sm_103a" in ck.version()


def test_library_is_built_for_sm_103a(ck):
    # the fatbin inside the shared object names the target architecture
    blob = open(ck.build.LIB, "rb").read()
    assert b"sm_103a" in blob


def test_host_isqrt(ck):
    rng = np.random.default_rng(21)
    vals = [0, 1, 2, 3, 42950, 42951, 2**32, 2**32 + 42950, 2**63, 2**64 - 1]
    for k in list(rng.integers(1, 2**32 - 1, 2000, dtype=np.uint64)) + [2**32 - 1, 2**31]:
        k = int(k)
        vals += [k * k - 1, k * k, k * k + 1]
    vals += [int(v) for v in rng.integers(0, 2**63, 2000, dtype=np.uint64)]
    for v in vals:
        assert ck.host_isqrt(v) == math.isqrt(v), v


def _trunc_div(n, d):
    q = abs(n) // d
    return q if n >= 0 else -q


def test_host_division_by_invariant_divisor(ck):
    rng = np.random.default_rng(22)
    divisors = [1, 2, 3, 5, 7, 207, 208, 255, 256, 257, 65535, 65536, 65537, 2**31 - 1, 2**31,
                2**32 - 1] + [int(v) for v in rng.integers(1, 2**32, 300, dtype=np.uint64)]
    numerators = [0, 1, -1, 2**63 - 1, -2**63, -2**63 + 1, 2**62, -(256 * 207 + 1)]
    numerators += [int(v) for v in rng.integers(-2**63, 2**63 - 1, 200, dtype=np.int64)]
    numerators += [int(v) for v in rng.integers(-2**40, 2**40, 200, dtype=np.int64)]
    for d in divisors:
        for n in numerators + [d * 12345 - 1, -d * 12345 + 1, d, -d, d - 1, -(d - 1)]:
            n = max(min(n, 2**63 - 1), -2**63)
            assert ck.host_div_trunc(n, d) == _trunc_div(n, d), (n, d)


def test_host_division_reciprocal_for_every_small_divisor_and_near_powers_of_two(ck):
    """The reciprocal the normalization builds from two estimated 64-by-32 divisions: every
    divisor up to 5,000 and those next to each power of two, each against numerators at the
    quotient boundaries and the extremes."""
    divisors = list(range(1, 5001))
    for k in range(1, 33):
        divisors += [v for v in (2**k - 1, 2**k, 2**k + 1) if 1 <= v < 2**32]
    for d in divisors:
        for n in (0, d - 1, d, 2**63 - 1, -2**63, d * (2**31 // d) - 1, 12345 * d + d - 1, -(d + 1)):
            n = max(min(n, 2**63 - 1), -2**63)
            assert ck.host_div_trunc(n, d) == _trunc_div(n, d), (n, d)


def test_host_probability_from_a_reciprocal_estimate(ck):
    """The attention probability floor((e << 24) / z) as the kernels form it: sums from one
    table entry (2^30) to 2^46 - 1, exponentials (table entries, at most 2^30 and at most the
    sum) from 0 up, at the quotient boundaries."""
    rng = np.random.default_rng(23)
    sums = [2**30, 2**30 + 1, 2**31 - 1, 2**31, 3 * 2**30 + 7, 2**40 - 1, 2**43, 2**46 - 1]
    sums += [int(v) for v in rng.integers(2**30, 2**46, 300, dtype=np.uint64)]
    for z in sums:
        top = min(z, 2**30)  # an exponential is one table entry, at most 2^30
        es = [0, 1, top, top - 1] + [int(v) for v in rng.integers(0, top + 1, 20)]
        for k in (1, 2, 3, 1000):  # just below and at multiples of z / 2^24
            q = k * z >> 24
            es += [e for e in ((q * z + 2**24 - 1) >> 24, (q * z) >> 24) if 0 <= e <= min(z, 2**30)]
        for e in es:
            assert ck.host_probability(e, z) == (e << 24) // z, (e, z)


def test_library_fails_loudly_without_a_gpu(ck):
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    # the product path has no CPU fallback: a model cannot be loaded without a device
    import synth
    with pytest.raises(Exception):
        ck.Model.load(synth.build_artifact(synth.TINY_WS))


# ---------------------------------------------------------------- tokenizer (host code)

def test_library_tokenizer_matches_the_oracle():
    """The library's phases 0 to 2 and token text against the oracle's, on seeded prompts
    over synthetic vocabularies (host code: no GPU needed)."""
    import fixed_point_int8_gb300 as ck
    import oracle
    import synth
    for n, seed in ((512, 0x5EED0011), (32000, 0x5EED0003)):
        blob = synth.tokenizer_blob(n, seed)
        rc, tok = ck.Tokenizer.load(blob, n)
        assert rc == 0
        v = oracle.Vocab(blob, n)
        for run in range(8):
            text = synth.prompt_text(120, seed, run, blob)
            rco, want = v.encode(text)
            rcg, got = tok.encode(text)
            assert rco == rcg == 0 and got.tolist() == want, run
            rc, back = tok.decode(got)
            assert rc == 0 and back == v.decode(want) == text
            ids = [int(x) for x in synth.random_u32(40, seed, 77 + run, 0, n - 1)]
            assert tok.decode(ids, prev=1)[1] == v.decode(ids, prev=1)
        for bad in (b"a\x00b", b"\xff", b"\xed\xa0\x80", b"x" * 1025):   # zero, bad lead, surrogate, long
            assert tok.encode(bad)[0] == v.encode(bad)[0] == 6
        assert tok.encode(b"")[1].tolist() == v.encode(b"")[1] == [1]
    blob = synth.tokenizer_blob(512, 1)
    assert ck.Tokenizer.load(blob[:100], 512)[0] == 2                     # truncated
    import struct
    dup = struct.pack("<I", 1) + struct.pack("<fi", 0.0, 1) + b"a" + struct.pack("<fi", 0.0, 1) + b"a"
    assert ck.Tokenizer.load(dup, 2)[0] == 2                               # a repeated string
    with pytest.raises(ValueError):
        oracle.Vocab(dup, 2)


# ---------------------------------------------------------------- the page's state (host code)

def test_page_converters_reject_wrong_inputs():
    import fixed_point_int8_gb300 as ck
    lib = ck.lib()
    assert lib.ck_page_size(None, 1, 1, None) == 10
    assert lib.ck_state_from_page(None, None, 0, None, 0) == 10
