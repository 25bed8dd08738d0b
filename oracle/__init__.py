"""ORACLE — test infrastructure, not part of the product.

Python binding of ``ck_oracle.c``, the plain CPU restatement of curta-core's integer
forward pass (page "The inference core", curta.chat docs).  Only ``tests/``,
``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline leg may import this package.
It imports nothing from the GPU library and the library imports nothing from it.

Pin status (each function is checked in ``tests/test_oracle_pins.py`` against values the
page fixes, closed forms, textbook routines or brute force):
  isqrt, embed, rmsnorm, matrow, fits32, rotate, attention_head, silu, silu_gate, argmax,
  xorshift_next, sample_index, draw_walk, sample, page_state_size, Vocab (tokenizer phases
  0 to 2 and token text): pinned.
  Whole-model token streams: parity unpinned against curta-core itself (the page prints no
  tokens or logits for a model); pinned only through the per-step pins and invariants.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "ck_oracle.c")
_LIB = os.path.join(_HERE, "_oracle.so")
_lib = None

EVENT_NAMES = ("matrow_acc", "matrow_scale", "norm_squares", "norm_product", "rotary",
               "score_dot", "score_scale", "silu_product", "residual")
LAYOUT_NAMES = ("prompt", "out", "x", "xb", "q", "o", "y", "h", "logits", "scores", "k", "v", "size")

# header offsets of the ids-mode state (format "CKSTATE1")
H_PHASE, H_POSITION, H_NPROMPT, H_MAXTOK, H_CACHE, H_GENERATED = 8, 12, 16, 20, 24, 28
H_FLAGS, H_TEMP, H_ERROR, H_LASTTOK, H_SEED, H_TURNS, H_ERRKEY, H_MAXLOGIT = 32, 36, 40, 44, 48, 56, 64, 72
H_EXPSUM, H_DRAW = 112, 120
PHASE_RUNNING, PHASE_DONE, PHASE_FAILED = 3, 20, 21
FLAG_STOP_TOKENS = 1


def build(force: bool = False) -> str:
    """Compile ``ck_oracle.c`` into ``_oracle.so`` (gcc -O2, OpenMP over independent rows)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-fPIC", "-shared", "-fopenmp", "-o", tmp, _SRC])
        os.replace(tmp, _LIB)
    return _LIB


class TurnResult(ctypes.Structure):
    _fields_ = [(n, ctypes.c_uint32) for n in (
        "complete", "generated", "generated_this_turn", "token", "work",
        "err_position", "err_layer", "err_phase", "err_element")]

    def as_dict(self) -> dict:
        return {n: int(getattr(self, n)) for n, _ in self._fields_}


def _lib_():
    global _lib
    if _lib is None:
        lib = ctypes.CDLL(build())
        vp, u32, u64, i64, i32 = ctypes.c_void_p, ctypes.c_uint32, ctypes.c_uint64, ctypes.c_int64, ctypes.c_int32
        sig = {
            "orc_isqrt": ([u64], u64),
            "orc_embed": ([vp, u32, u32, vp], None),
            "orc_rmsnorm": ([vp, vp, u32, vp], None),
            "orc_matrow": ([vp, u64, vp, u32, u32, vp, vp], None),
            "orc_fits32": ([i64], ctypes.c_int),
            "orc_rotate": ([i64, i64, i32, i32, vp, vp], None),
            "orc_attention_head": ([vp, vp, vp, u64, u32, u32, u32, vp, vp, vp], None),
            "orc_silu": ([i64, vp], i64),
            "orc_silu_gate": ([vp, vp, u32, vp, vp], None),
            "orc_argmax": ([vp, u32], u32),
            "orc_xorshift_next": ([ctypes.POINTER(u64)], u64),
            "orc_sample_index": ([i64, i64, u32], u32),
            "orc_draw_walk": ([vp, u32, u64], u32),
            "orc_sample": ([vp, u32, u32, vp, ctypes.POINTER(u64), ctypes.POINTER(i64),
                            ctypes.POINTER(u64), ctypes.POINTER(u64)], u32),
            "orc_page_state_size": ([vp, u32, u32], u64),
            "orc_model_open": ([vp, u64, ctypes.POINTER(vp)], ctypes.c_int),
            "orc_model_close": ([vp], None),
            "orc_state_size": ([vp, u32, u32], u64),
            "orc_init_state": ([vp, vp, u64, vp, u32, u32, u32, u64, u32], ctypes.c_int),
            "orc_turn": ([vp, vp, u64, u32, ctypes.POINTER(TurnResult)], ctypes.c_int),
            "orc_state_layout": ([vp, u32, u32, vp], None),
            "orc_events_reset": ([ctypes.c_int], None),
            "orc_events_get": ([vp], None),
            "orc_threads": ([], ctypes.c_int),
            "orc_vocab_open": ([vp, u64, u32, ctypes.POINTER(vp)], ctypes.c_int),
            "orc_vocab_close": ([vp], None),
            "orc_vocab_lookup": ([vp, vp, u32], i64),
            "orc_encode": ([vp, vp, u32, vp, u32, ctypes.POINTER(u32)], ctypes.c_int),
            "orc_decode_piece": ([vp, u32, u32, vp, u32], u32),
            "orc_page_size": ([vp, u32, u32], u64),
            "orc_page_layout_of": ([vp, u32, u32, vp], None),
            "orc_page_init": ([vp, vp, u64, vp, u32, u32, u32, u64], ctypes.c_int),
            "orc_page_turn": ([vp, vp, vp, u64, u32, ctypes.POINTER(u32)], ctypes.c_int),
        }
        for name, (args, res) in sig.items():
            f = getattr(lib, name)
            f.argtypes = args
            f.restype = res
        _lib = lib
    return _lib


def _c(a: np.ndarray, dtype) -> np.ndarray:
    return np.ascontiguousarray(a, dtype=dtype)


# ------------------------------------------------------------------ single steps

def isqrt(v: int) -> int:
    return int(_lib_().orc_isqrt(v))


def embed(row: np.ndarray, scale: int) -> np.ndarray:
    row = _c(row, np.uint8)
    out = np.zeros(row.size, dtype=np.int64)
    _lib_().orc_embed(row.ctypes.data, scale, row.size, out.ctypes.data)
    return out


def rmsnorm(x: np.ndarray, w: np.ndarray) -> np.ndarray:
    x, w = _c(x, np.int64), _c(w, np.int32)
    assert x.size == w.size and x.size > 0
    out = np.zeros(x.size, dtype=np.int64)
    _lib_().orc_rmsnorm(x.ctypes.data, w.ctypes.data, x.size, out.ctypes.data)
    return out


def matrow(W: np.ndarray, scale: np.ndarray, x: np.ndarray, cols: int | None = None) -> np.ndarray:
    """W is [rows][pitch] uint8; the first ``cols`` (default pitch) columns are used."""
    W, scale, x = _c(W, np.uint8), _c(scale, np.uint32), _c(x, np.int64)
    rows, pitch = W.shape
    cols = pitch if cols is None else cols
    assert x.size >= cols and scale.size >= rows
    out = np.zeros(rows, dtype=np.int64)
    _lib_().orc_matrow(W.ctypes.data, pitch, scale.ctypes.data, rows, cols, x.ctypes.data, out.ctypes.data)
    return out


def fits32(v: int) -> bool:
    return bool(_lib_().orc_fits32(v))


def rotate(a: int, b: int, c: int, s: int) -> tuple[int, int]:
    a2, b2 = ctypes.c_int64(), ctypes.c_int64()
    _lib_().orc_rotate(a, b, c, s, ctypes.byref(a2), ctypes.byref(b2))
    return a2.value, b2.value


def attention_head(q: np.ndarray, K: np.ndarray, V: np.ndarray, inv: int, exp_tab: np.ndarray):
    """q i64[hd]; K, V i32[p][hd].  Returns (out i64[hd], probabilities i64[p])."""
    q, K, V, e = _c(q, np.int64), _c(K, np.int32), _c(V, np.int32), _c(exp_tab, np.uint32)
    p, hd = K.shape
    scores = np.zeros(p, dtype=np.int64)
    out = np.zeros(hd, dtype=np.int64)
    _lib_().orc_attention_head(q.ctypes.data, K.ctypes.data, V.ctypes.data, hd, p, hd, inv,
                               e.ctypes.data, scores.ctypes.data, out.ctypes.data)
    return out, scores


def silu(g: int, tab: np.ndarray) -> int:
    tab = _c(tab, np.int32)
    return int(_lib_().orc_silu(g, tab.ctypes.data))


def silu_gate(g: np.ndarray, u: np.ndarray, tab: np.ndarray) -> np.ndarray:
    g, u, tab = _c(g, np.int64), _c(u, np.int64), _c(tab, np.int32)
    out = np.zeros(g.size, dtype=np.int64)
    _lib_().orc_silu_gate(g.ctypes.data, u.ctypes.data, g.size, tab.ctypes.data, out.ctypes.data)
    return out


def argmax(logits: np.ndarray) -> int:
    logits = _c(logits, np.int64)
    return int(_lib_().orc_argmax(logits.ctypes.data, logits.size))


def xorshift_next(state: int) -> tuple[int, int]:
    """One step of the sampling generator: returns (new state, output)."""
    s = ctypes.c_uint64(state)
    out = int(_lib_().orc_xorshift_next(ctypes.byref(s)))
    return int(s.value), out


def sample_index(m: int, l: int, temperature_q16: int) -> int:
    return int(_lib_().orc_sample_index(m, l, temperature_q16))


def draw_walk(e: np.ndarray, r: int) -> int:
    e = _c(e, np.uint64)
    return int(_lib_().orc_draw_walk(e.ctypes.data, e.size, r))


def sample(logits: np.ndarray, temperature_q16: int, exp_tab: np.ndarray, state: int) -> dict:
    """Phase 19 on a logit vector: {token, state, max, sum, draw}."""
    logits, e = _c(logits, np.int64), _c(exp_tab, np.uint32)
    s, m, z, d = ctypes.c_uint64(state), ctypes.c_int64(), ctypes.c_uint64(), ctypes.c_uint64()
    tok = _lib_().orc_sample(logits.ctypes.data, logits.size, temperature_q16, e.ctypes.data,
                             ctypes.byref(s), ctypes.byref(m), ctypes.byref(z), ctypes.byref(d))
    return {"token": int(tok), "state": int(s.value), "max": int(m.value), "sum": int(z.value),
            "draw": int(d.value)}


def page_state_size(config, prompt_bytes: int, max_tokens: int) -> int:
    cfg = np.array(config, dtype=np.uint32)
    return int(_lib_().orc_page_state_size(cfg.ctypes.data, prompt_bytes, max_tokens))


def threads() -> int:
    """OpenMP threads the oracle's row loops use."""
    return int(_lib_().orc_threads())


def events_reset(enable: bool = True) -> None:
    _lib_().orc_events_reset(1 if enable else 0)


def events() -> dict:
    out = np.zeros(len(EVENT_NAMES), dtype=np.uint64)
    _lib_().orc_events_get(out.ctypes.data)
    return {n: int(v) for n, v in zip(EVENT_NAMES, out)}


# ------------------------------------------------------------------ whole model

class Model:
    """A parsed artifact; the array must stay alive (the oracle aliases it)."""

    def __init__(self, artifact: np.ndarray):
        self.artifact = _c(artifact, np.uint8)
        h = ctypes.c_void_p()
        rc = _lib_().orc_model_open(self.artifact.ctypes.data, self.artifact.size, ctypes.byref(h))
        if rc:
            raise ValueError(f"oracle: artifact rejected with error {rc}")
        self._h = h
        self.config = tuple(int(v) for v in self.artifact[8:36].view("<u4"))

    def close(self):
        if self._h:
            _lib_().orc_model_close(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def state_size(self, n_prompt: int, max_tokens: int) -> int:
        return int(_lib_().orc_state_size(self._h, n_prompt, max_tokens))

    def layout(self, n_prompt: int, max_tokens: int) -> dict:
        out = np.zeros(13, dtype=np.uint64)
        _lib_().orc_state_layout(self._h, n_prompt, max_tokens, out.ctypes.data)
        return {n: int(v) for n, v in zip(LAYOUT_NAMES, out)}

    def init_state(self, ids, max_tokens: int, temperature_q16: int = 0, seed: int = 0,
                   flags: int = 0, length: int | None = None):
        """Returns (rc, state bytes)."""
        ids = _c(np.asarray(ids), np.uint32)
        n = self.state_size(max(ids.size, 1), max(max_tokens, 1)) if length is None else length
        st = np.zeros(max(n, 256), dtype=np.uint8)
        rc = _lib_().orc_init_state(self._h, st.ctypes.data, n, ids.ctypes.data, ids.size,
                                    max_tokens, temperature_q16, seed, flags)
        return rc, st

    def turn(self, state: np.ndarray, n_positions: int):
        """Runs up to n_positions positions in place.  Returns (rc, result dict)."""
        assert state.dtype == np.uint8 and state.flags.c_contiguous
        res = TurnResult()
        rc = _lib_().orc_turn(self._h, state.ctypes.data, state.size, n_positions, ctypes.byref(res))
        return rc, res.as_dict()


class Vocab:
    """A tokenizer vocabulary (llama2.c's tokenizer file layout) of n tokens."""

    def __init__(self, blob: bytes, n: int):
        self.blob = np.frombuffer(bytes(blob), dtype=np.uint8).copy()
        h = ctypes.c_void_p()
        rc = _lib_().orc_vocab_open(self.blob.ctypes.data, self.blob.size, n, ctypes.byref(h))
        if rc:
            raise ValueError(f"oracle: vocabulary rejected with error {rc}")
        self._h = h
        self.n = n

    def __del__(self):
        try:
            if self._h:
                _lib_().orc_vocab_close(self._h)
        except Exception:
            pass

    def lookup(self, s: bytes) -> int:
        b = np.frombuffer(bytes(s) or b"\0", dtype=np.uint8)
        return int(_lib_().orc_vocab_lookup(self._h, b.ctypes.data, len(s)))

    def encode(self, text: bytes):
        """Phases 0 to 2.  Returns (rc, ids)."""
        t = np.frombuffer(bytes(text) or b"\0", dtype=np.uint8)
        cap = len(text) + 2
        ids = np.zeros(cap, dtype=np.uint32)
        n = ctypes.c_uint32()
        rc = _lib_().orc_encode(self._h, t.ctypes.data, len(text), ids.ctypes.data, cap, ctypes.byref(n))
        return rc, ids[:n.value].tolist() if rc == 0 else []

    def piece(self, prev: int, tok: int) -> bytes:
        out = np.zeros(1024, dtype=np.uint8)
        n = _lib_().orc_decode_piece(self._h, prev, tok, out.ctypes.data, out.size)
        return out[:n].tobytes()

    def decode(self, ids, prev: int = 0) -> bytes:
        """The text of the tokens ids, each after the one before it (prev before the first)."""
        out = b""
        for t in ids:
            out += self.piece(prev, int(t))
            prev = int(t)
        return out


PAGE_LAYOUT_NAMES = ("prompt", "ptok", "out", "text", "x", "w0", "w1", "w2", "gate", "up", "logits",
                     "scores", "k", "v", "size", "cache")


def page_new(model: "Model", prompt: bytes, max_tokens: int, temperature_q16: int = 0, seed: int = 0):
    """A fresh page state ("CURTAST2") for a text prompt.  Returns (rc, state bytes)."""
    n = int(_lib_().orc_page_size(model._h, len(prompt), max_tokens))
    st = np.zeros(n, dtype=np.uint8)
    p = np.frombuffer(bytes(prompt) or b"\0", dtype=np.uint8)
    rc = _lib_().orc_page_init(model._h, st.ctypes.data, n, p.ctypes.data, len(prompt), max_tokens,
                               temperature_q16, seed)
    return rc, st


def page_layout(model: "Model", prompt_bytes: int, max_tokens: int) -> dict:
    out = np.zeros(16, dtype=np.uint64)
    _lib_().orc_page_layout_of(model._h, prompt_bytes, max_tokens, out.ctypes.data)
    return {k: int(v) for k, v in zip(PAGE_LAYOUT_NAMES, out)}


def page_turn(model: "Model", vocab: "Vocab", state: np.ndarray, n_steps: int):
    """Up to n_steps phase steps in place.  Returns (rc, steps run)."""
    steps = ctypes.c_uint32()
    rc = _lib_().orc_page_turn(model._h, vocab._h, state.ctypes.data, state.size, n_steps, ctypes.byref(steps))
    return rc, int(steps.value)


def page_header(state: np.ndarray) -> dict:
    u32 = lambda o: int(state[o:o + 4].view("<u4")[0])
    u64 = lambda o: int(state[o:o + 8].view("<u8")[0])
    return {"phase": u32(8), "layer": u32(12), "row": u32(16), "position": u32(20), "token": u32(24),
            "prompt_bytes": u32(28), "prompt_tokens": u32(32), "max_tokens": u32(36), "temperature": u32(40),
            "generated": u32(44), "text_bytes": u32(48), "generator": u64(72), "turns": u64(80),
            "max_score": int(state[88:96].view("<i8")[0]), "chosen": u32(96), "exp_sum": u64(104),
            "draw": u64(112), "att_stage": u32(120), "att_index": u32(124)}


def header(state: np.ndarray) -> dict:
    u32 = lambda o: int(state[o:o + 4].view("<u4")[0])
    u64 = lambda o: int(state[o:o + 8].view("<u8")[0])
    return {"phase": u32(H_PHASE), "position": u32(H_POSITION), "n_prompt": u32(H_NPROMPT),
            "max_tokens": u32(H_MAXTOK), "cache": u32(H_CACHE), "generated": u32(H_GENERATED),
            "flags": u32(H_FLAGS), "temperature": u32(H_TEMP), "error": u32(H_ERROR),
            "last_token": u32(H_LASTTOK), "generator": u64(H_SEED), "turns": u64(H_TURNS),
            "err_key": u64(H_ERRKEY), "exp_sum": u64(H_EXPSUM), "draw": u64(H_DRAW),
            "max_logit": int(state[H_MAXLOGIT:H_MAXLOGIT + 8].view("<i8")[0])}
