"""Seeded synthetic inputs shared by the CPU oracle and the GPU library.

This module only draws random integers (through ``synth.c``) and lays them out in the
model-artifact format that ``include/ck.h`` documents.  It holds none of the forward
pass's arithmetic.  The exponential, SiLU and rotary tables are built here in double
precision because on the curta-core page they are inputs computed once at conversion
("The inference core", section "Lookup tables"); both sides read them from the artifact.

Input recipe (all integers, all from xorshift64* streams, see ``synth.c``):
  * weight bytes uniform 0..255 (a weight is the byte minus 128);
  * row scales: ``literal`` rule uniform in [0.9, 1.1] x 2^21 (about 2^24 / 8), or the
    ``well`` rule uniform in [0.75, 1.25] x 2^24 / (74 sqrt(cols)) so that a matrix row
    maps unit-RMS inputs to unit-RMS outputs (74 is the RMS of a uniform byte minus 128);
    embedding rows under ``well`` use 2^24 / 74 so embedded vectors have unit RMS;
  * norm weights uniform in [0.9, 1.1] x 2^24;
  * prompt ids uniform in [3, vocab).
"""
from __future__ import annotations

import ctypes
import math
import os
import subprocess
from dataclasses import dataclass, field

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "synth.c")
_LIB = os.path.join(_HERE, "_synth.so")
_lib = None

MAGIC = b"CKMODEL1"
HEADER_BYTES = 64
TABLE_ENTRIES = 4097
TENSOR_ALIGN = 64
FLAG_TIED = 1

# Tensor directory order of the artifact (see include/ck.h).
T_EMBED, T_EMBED_SCALE, T_FINAL_NORM, T_CLS, T_CLS_SCALE, T_ROPE, T_EXP, T_SILU = range(8)
GLOBAL_TENSORS = 8
PER_LAYER = 16
(L_ATTN_NORM, L_WQ, L_SQ, L_WK, L_SK, L_WV, L_SV, L_WO, L_SO, L_FFN_NORM, L_W1, L_S1,
 L_W3, L_S3, L_W2, L_S2) = range(PER_LAYER)

# Stream ids for draws that are not artifact tensors.
STREAM_PROMPT = 1_000_000
STREAM_VECTOR = 2_000_000
STREAM_MATRIX = 3_000_000


def build(force: bool = False) -> str:
    """Compile ``synth.c`` into ``_synth.so`` beside it (gcc, OpenMP over rows)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-fPIC", "-shared", "-fopenmp", "-o", tmp, _SRC])
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    if _lib is None:
        lib = ctypes.CDLL(build())
        u64, u32, i64, vp = ctypes.c_uint64, ctypes.c_uint32, ctypes.c_int64, ctypes.c_void_p
        lib.synth_xs64s_next.argtypes = [ctypes.POINTER(u64)]
        lib.synth_xs64s_next.restype = u64
        lib.synth_stream_seed.argtypes = [u64, u32, u64]
        lib.synth_stream_seed.restype = u64
        lib.synth_bytes.argtypes = [vp, u64, u64, u64, u64, u32]
        lib.synth_u32_range.argtypes = [vp, u64, u64, u32, u32, u32]
        lib.synth_i64_range.argtypes = [vp, u64, u64, u32, i64, i64]
        _lib = lib
    return _lib


def xs64s_sequence(seed: int, n: int) -> list[int]:
    """n successive xorshift64* outputs from ``seed`` (0 starts at 0x9E3779B97F4A7C15)."""
    lib = _load()
    st = ctypes.c_uint64(seed)
    return [int(lib.synth_xs64s_next(ctypes.byref(st))) for _ in range(n)]


def random_bytes(rows: int, cols: int, seed: int, tensor: int, pitch: int | None = None) -> np.ndarray:
    pitch = cols if pitch is None else pitch
    out = np.zeros((rows, pitch), dtype=np.uint8)
    if rows and cols:
        _load().synth_bytes(out.ctypes.data, rows, cols, pitch, seed, tensor)
    return out


def random_u32(n: int, seed: int, tensor: int, lo: int, hi: int) -> np.ndarray:
    assert 0 <= lo <= hi < 2**32
    out = np.zeros(n, dtype=np.uint32)
    if n:
        _load().synth_u32_range(out.ctypes.data, n, seed, tensor, lo, hi)
    return out


def random_i64(n: int, seed: int, tensor: int, lo: int, hi: int) -> np.ndarray:
    assert -2**63 <= lo <= hi < 2**63
    out = np.zeros(n, dtype=np.int64)
    if n:
        _load().synth_i64_range(out.ctypes.data, n, seed, tensor, lo, hi)
    return out


# ----------------------------------------------------------------------------- tables

def _round_half_away(v: float) -> int:
    return int(math.floor(v + 0.5)) if v >= 0 else -int(math.floor(-v + 0.5))


def exp_table() -> np.ndarray:
    """4,097 entries of e^(-i/256) with 30 fractional bits (u32)."""
    return np.array([_round_half_away(math.exp(-i / 256.0) * 2.0**30) for i in range(TABLE_ENTRIES)],
                    dtype=np.uint32)


def silu_table() -> np.ndarray:
    """4,097 entries of silu(i/128 - 16) with 16 fractional bits (i32)."""
    vals = []
    for i in range(TABLE_ENTRIES):
        x = i / 128.0 - 16.0
        vals.append(_round_half_away(x / (1.0 + math.exp(-x)) * 2.0**16))
    return np.array(vals, dtype=np.int32)


def rope_table(context: int, head_dim: int) -> np.ndarray:
    """[context][head_dim/2][2] (cos, sin) with 24 fractional bits, theta_j = 10000^(-2j/hd)."""
    half = head_dim // 2
    out = np.zeros((context, half, 2), dtype=np.int32)
    for j in range(half):
        theta = 10000.0 ** (-2.0 * j / head_dim)
        for p in range(context):
            out[p, j, 0] = _round_half_away(math.cos(p * theta) * 2.0**24)
            out[p, j, 1] = _round_half_away(math.sin(p * theta) * 2.0**24)
    return out


def inv_sqrt_head(head_dim: int) -> int:
    return _round_half_away(2.0**24 / math.sqrt(head_dim))


# ----------------------------------------------------------------------------- models

@dataclass(frozen=True)
class ModelSpec:
    name: str
    dim: int
    hidden: int
    layers: int
    heads: int
    kv_heads: int
    vocab: int
    context: int
    scale_rule: str = "well"      # "well" or "literal"
    tied: bool = True
    seed: int = 0x5EED0000

    @property
    def head_dim(self) -> int:
        return self.dim // self.heads

    @property
    def kv_dim(self) -> int:
        return self.head_dim * self.kv_heads

    def config(self) -> tuple[int, ...]:
        return (self.dim, self.hidden, self.layers, self.heads, self.kv_heads, self.vocab, self.context)

    def weight_bytes_per_token(self) -> int:
        """Bytes of weights one generating position streams (classifier included)."""
        d, h, kv = self.dim, self.hidden, self.kv_dim
        per_layer = d * d * 2 + kv * d * 2 + h * d * 3
        return self.layers * per_layer + self.vocab * d


@dataclass(frozen=True)
class Workload:
    spec: ModelSpec
    n_prompt: int
    steps: int
    runs: int = 1


# Seeds follow 0x5EED0000 + config number (1-based as the workload list numbers them).
TINY = ModelSpec("tiny", 64, 172, 2, 4, 4, 512, 32, scale_rule="literal", seed=0x5EED0001)
TINY_WS = ModelSpec("tiny_ws", 64, 172, 2, 4, 4, 512, 32, scale_rule="well", tied=False, seed=0x5EED0011)
GQA = ModelSpec("gqa_stories260k_shape", 64, 172, 5, 8, 4, 512, 512, scale_rule="well", tied=False, seed=0x5EED0021)
GQA_TIED = ModelSpec("gqa_tied", 64, 172, 5, 8, 4, 512, 512, scale_rule="well", tied=True, seed=0x5EED0022)
LLAMA7B = ModelSpec("llama7b_shape", 4096, 11008, 32, 32, 32, 32000, 2048, tied=False, seed=0x5EED0003)
ONE_B = ModelSpec("1b_shape", 2048, 5632, 22, 32, 32, 32000, 2048, tied=False, seed=0x5EED0004)
ONE_B_LONG = ModelSpec("1b_shape_ctx8192", 2048, 5632, 22, 32, 32, 32000, 8192, tied=False, seed=0x5EED0005)

WORKLOADS = {
    "tiny": Workload(TINY, 8, 16),
    "tiny_ws": Workload(TINY_WS, 8, 16),
    "gqa": Workload(GQA, 12, 40),
    "gqa_tied": Workload(GQA_TIED, 5, 20),
    "7b": Workload(LLAMA7B, 128, 256),
    "1b_x64": Workload(ONE_B, 64, 128, runs=64),
    "1b_long": Workload(ONE_B_LONG, 7936, 256),
}

MATROW_SHAPES = [(4096, 4096), (11008, 4096), (4096, 11008), (32000, 4096)]
MATROW_SEED = 0x5EED0002


def _align(n: int, a: int = TENSOR_ALIGN) -> int:
    return (n + a - 1) // a * a


def tensor_shapes(spec: ModelSpec) -> list[tuple[str, tuple[int, ...]]]:
    """(dtype, shape) of each artifact tensor in directory order."""
    d, h, v, kv, hd = spec.dim, spec.hidden, spec.vocab, spec.kv_dim, spec.head_dim
    out = [("u8", (v, d)), ("u32", (v,)), ("i32", (d,)),
           ("u8", (0, d) if spec.tied else (v, d)), ("u32", (0,) if spec.tied else (v,)),
           ("i32", (spec.context, hd // 2, 2)), ("u32", (TABLE_ENTRIES,)), ("i32", (TABLE_ENTRIES,))]
    for _ in range(spec.layers):
        out += [("i32", (d,)), ("u8", (d, d)), ("u32", (d,)), ("u8", (kv, d)), ("u32", (kv,)),
                ("u8", (kv, d)), ("u32", (kv,)), ("u8", (d, d)), ("u32", (d,)), ("i32", (d,)),
                ("u8", (h, d)), ("u32", (h,)), ("u8", (h, d)), ("u32", (h,)), ("u8", (d, h)), ("u32", (d,))]
    return out


_ITEM = {"u8": 1, "u32": 4, "i32": 4}
_NP = {"u8": np.uint8, "u32": np.uint32, "i32": np.int32}


def _scale_bounds(spec: ModelSpec, cols: int, embedding: bool) -> tuple[int, int]:
    if spec.scale_rule == "literal":
        base = 2.0**21
        return _round_half_away(0.9 * base), _round_half_away(1.1 * base)
    base = 2.0**24 / 74.0 if embedding else 2.0**24 / (74.0 * math.sqrt(cols))
    return max(1, _round_half_away(0.75 * base)), max(1, _round_half_away(1.25 * base))


def build_artifact(spec: ModelSpec) -> np.ndarray:
    """The whole model artifact as one uint8 array (layout in include/ck.h)."""
    shapes = tensor_shapes(spec)
    n = len(shapes)
    off = _align(HEADER_BYTES + 16 * n)
    entries = []
    for dt, shp in shapes:
        length = int(np.prod(shp)) * _ITEM[dt]
        entries.append((off if length else 0, length))
        off = _align(off + length)
    total = off
    art = np.zeros(total, dtype=np.uint8)
    hdr = art[:HEADER_BYTES]
    hdr[:8] = np.frombuffer(MAGIC, dtype=np.uint8)
    hdr[8:36] = np.frombuffer(np.array(spec.config(), dtype="<u4").tobytes(), dtype=np.uint8)
    tail = np.array([inv_sqrt_head(spec.head_dim), FLAG_TIED if spec.tied else 0, n], dtype="<u4")
    hdr[36:48] = np.frombuffer(tail.tobytes(), dtype=np.uint8)
    hdr[48:56] = np.frombuffer(np.array([total], dtype="<u8").tobytes(), dtype=np.uint8)
    dirarr = np.array(entries, dtype="<u8").reshape(-1)
    art[HEADER_BYTES:HEADER_BYTES + 16 * n] = np.frombuffer(dirarr.tobytes(), dtype=np.uint8)

    def view(i):
        dt, shp = shapes[i]
        o, length = entries[i]
        return art[o:o + length].view(_NP[dt]).reshape(shp)

    seed = spec.seed
    lib = _load()

    def fill_bytes(i):
        a = view(i)
        if a.size:
            lib.synth_bytes(a.ctypes.data, a.shape[0], a.shape[1], a.shape[1], seed, i)

    def fill_scales(i, cols, embedding=False):
        a = view(i)
        lo, hi = _scale_bounds(spec, cols, embedding)
        if a.size:
            lib.synth_u32_range(a.ctypes.data, a.size, seed, i, lo, hi)

    def fill_norm(i):
        a = view(i)
        lo, hi = _round_half_away(0.9 * 2**24), _round_half_away(1.1 * 2**24)
        lib.synth_u32_range(a.ctypes.data, a.size, seed, i, lo, hi)   # < 2^31: same bits as i32

    fill_bytes(T_EMBED)
    fill_scales(T_EMBED_SCALE, spec.dim, embedding=True)
    fill_norm(T_FINAL_NORM)
    if not spec.tied:
        fill_bytes(T_CLS)
        fill_scales(T_CLS_SCALE, spec.dim)
    view(T_ROPE)[...] = rope_table(spec.context, spec.head_dim)
    view(T_EXP)[...] = exp_table()
    view(T_SILU)[...] = silu_table()
    for layer in range(spec.layers):
        b = GLOBAL_TENSORS + PER_LAYER * layer
        fill_norm(b + L_ATTN_NORM)
        fill_norm(b + L_FFN_NORM)
        for w, s, cols in ((L_WQ, L_SQ, spec.dim), (L_WK, L_SK, spec.dim), (L_WV, L_SV, spec.dim),
                           (L_WO, L_SO, spec.dim), (L_W1, L_S1, spec.dim), (L_W3, L_S3, spec.dim),
                           (L_W2, L_S2, spec.hidden)):
            fill_bytes(b + w)
            fill_scales(b + s, cols)
    return art


def artifact_tensor(art: np.ndarray, index: int) -> np.ndarray:
    """A tensor of an artifact as a flat typed view, read back through the directory."""
    cfg = art[8:36].view("<u4")
    layers = int(cfg[2])
    spec = ModelSpec("view", *[int(c) for c in cfg], tied=bool(art[40:44].view("<u4")[0] & FLAG_TIED))
    shapes = tensor_shapes(spec)
    assert len(shapes) == GLOBAL_TENSORS + PER_LAYER * layers
    o, length = (int(v) for v in art[HEADER_BYTES + 16 * index:HEADER_BYTES + 16 * index + 16].view("<u8"))
    dt, shp = shapes[index]
    return art[o:o + length].view(_NP[dt]).reshape(shp)


def prompt_ids(spec: ModelSpec, n: int, run: int = 0) -> np.ndarray:
    return random_u32(n, spec.seed, STREAM_PROMPT + run, 3, spec.vocab - 1)


def matrow_case(rows: int, cols: int, seed: int = MATROW_SEED, pitch: int | None = None):
    """(W [rows][pitch] u8, scales u32 [rows] in [2^20, 2^24], x i64 [cols] in +-8.0)."""
    w = random_bytes(rows, cols, seed, STREAM_MATRIX + rows * 7 + cols, pitch)
    s = random_u32(rows, seed, STREAM_MATRIX + 1 + rows * 7 + cols, 2**20, 2**24)
    x = random_i64(cols, seed, STREAM_VECTOR + rows * 7 + cols, -8 * 2**16, 8 * 2**16)
    return w, s, x


# ---------------------------------------------------------------- synthetic tokenizer

STREAM_VOCAB = 4_000_000
STREAM_TEXT = 5_000_000
_VOCAB_CHARS = [bytes([c]) for c in range(0x20, 0x7F)] + [c.encode() for c in "éüñöç—€"]
_TEXT_CHARS = "abcdefghijklmnopqrstuvwxyz      ETAONISRH.,;:!?'-0123456789éüñöç—€日本"


def tokenizer_blob(vocab: int, seed: int) -> bytes:
    """A synthetic vocabulary of `vocab` tokens in llama2.c's tokenizer file layout (u32
    longest token, then per token f32 score, i32 length, bytes): <unk>, the opening and
    closing tokens, the 256 byte tokens <0x00>..<0xFF>, the printable ASCII characters and a
    few 2- and 3-byte characters, then merged tokens, each the concatenation of two earlier
    text tokens drawn from the seeded stream (at most 16 bytes, no repeats), with scores
    falling by 0.25 a token so earlier merges win.  Characters of the prompts it cannot
    spell (two CJK characters) fall back to byte tokens."""
    import struct
    toks = [(b"<unk>", 0.0), (b"\n<s>\n", 0.0), (b"\n</s>\n", 0.0)]
    toks += [(("<0x%02X>" % i).encode(), 0.0) for i in range(256)]
    text = [(c, -1e6) for c in _VOCAB_CHARS]
    toks += text[: max(0, vocab - len(toks))]
    seen = {t for t, _ in toks}
    pool = [t for t, _ in text]
    draws = xs64s_sequence(seed ^ STREAM_VOCAB, 8 * max(vocab, 64))
    k = 0
    score = -1.0
    while len(toks) < vocab and k + 1 < len(draws):
        a, b = pool[draws[k] % len(pool)], pool[draws[k + 1] % len(pool)]
        k += 2
        s = a + b
        if len(s) > 16 or s in seen:
            continue
        seen.add(s)
        toks.append((s, score))
        pool.append(s)
        score -= 0.25
    while len(toks) < vocab:  # draws ran out: filler tokens that no text spells
        s = ("<f%d>" % len(toks)).encode()
        toks.append((s, -1e9))
    out = struct.pack("<I", max(len(t) for t, _ in toks))
    for t, sc in toks:
        out += struct.pack("<fi", sc, len(t)) + t
    return out


def vocab_pieces(blob: bytes) -> list[bytes]:
    """The byte strings of a vocabulary in the tokenizer file layout."""
    import struct
    out, off = [], 4
    while off + 8 <= len(blob):
        _, n = struct.unpack_from("<fi", blob, off)
        out.append(blob[off + 8: off + 8 + n])
        off += 8 + n
    return out


def prompt_text(n_pieces: int, seed: int, run: int = 0, blob: bytes | None = None) -> bytes:
    """A seeded prompt: n_pieces pieces, each a single character (lower-case letters,
    spaces, capitals, digits, punctuation, 2- and 3-byte characters, two of them outside the
    synthetic vocabulary) or, with a vocabulary blob, half of the time one of its merged
    tokens, so that encoding it has merges to find."""
    d = xs64s_sequence(seed ^ STREAM_TEXT ^ (run << 20), 2 * n_pieces)
    merged = [t for t in vocab_pieces(blob)[259:] if len(t) > 1 and not t.startswith(b"<")] if blob else []
    out = b""
    for i in range(n_pieces):
        a, b = d[2 * i], d[2 * i + 1]
        if merged and a % 2:
            out += merged[b % len(merged)]
        else:
            out += _TEXT_CHARS[b % len(_TEXT_CHARS)].encode()
    return out
