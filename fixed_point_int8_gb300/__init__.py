"""fixed_point_int8_gb300 — GB300 (sm_103a) implementation of curta-core's bit-exact
fixed-point transformer forward pass.

This module is the thin Python binding of ``libck.so`` (the C ABI in ``include/ck.h``):
it only marshals arguments.  Every step of the forward pass runs in the library's CUDA
kernels; PyTorch supplies device memory and streams.  There is no CPU path: without the
built library (or a GPU) the calls fail.
"""
from __future__ import annotations

import ctypes
import os

import numpy as np

from . import build as _build

CK_FLAG_STOP_TOKENS = 1
PATH_AUTO, PATH_STEP, PATH_KERNELS = 0, 1, 2
PHASE_RUNNING, PHASE_DONE, PHASE_FAILED = 3, 20, 21
ERROR_NAMES = {1: "InvalidConfig", 2: "InvalidFormat", 3: "InvalidState", 4: "BufferTooSmall",
               5: "MissingWeights", 6: "InvalidPrompt", 7: "ContextExceeded", 8: "Arithmetic",
               9: "CudaError", 10: "InvalidArgument"}

_lib = None


class CkError(RuntimeError):
    def __init__(self, code: int, what: str):
        super().__init__(f"{what}: error {code} ({ERROR_NAMES.get(code, '?')})")
        self.code = code


class TurnResult(ctypes.Structure):
    _fields_ = [(n, ctypes.c_uint32) for n in (
        "complete", "generated", "generated_this_turn", "token", "work",
        "err_position", "err_layer", "err_phase", "err_element")]

    def as_dict(self) -> dict:
        return {n: int(getattr(self, n)) for n, _ in self._fields_}


class Config(ctypes.Structure):
    _fields_ = [(n, ctypes.c_uint32) for n in
                ("dim", "hidden", "layers", "heads", "kv_heads", "vocab", "context")]


def lib() -> ctypes.CDLL:
    """The loaded libck.so; raises if it has not been built."""
    global _lib
    if _lib is None:
        if not os.path.exists(_build.LIB):
            raise RuntimeError(f"libck.so is not built ({_build.LIB}); run fixed_point_int8_gb300.build.build()")
        L = ctypes.CDLL(_build.LIB)
        vp, sz, u32, u64, i64 = ctypes.c_void_p, ctypes.c_size_t, ctypes.c_uint32, ctypes.c_uint64, ctypes.c_int64
        sig = {
            "ck_model_size": ([vp, sz, ctypes.POINTER(sz)], ctypes.c_int),
            "ck_load_model": ([vp, sz, vp, sz, vp, ctypes.POINTER(vp)], ctypes.c_int),
            "ck_model_config": ([vp, ctypes.POINTER(Config)], ctypes.c_int),
            "ck_set_path": ([vp, ctypes.c_int], ctypes.c_int),
            "ck_set_step_slots": ([vp, ctypes.c_uint32], ctypes.c_int),
            "ck_set_attention_split": ([vp, ctypes.c_uint32], ctypes.c_int),
            "ck_set_step_prefetch": ([vp, ctypes.c_uint32], ctypes.c_int),
            "ck_set_step_wait_limit": ([vp, ctypes.c_uint32], ctypes.c_int),
            "ck_set_prefill": ([vp, ctypes.c_uint32], ctypes.c_int),
            "ck_free_model": ([vp], None),
            "ck_state_size": ([vp, u32, u32, ctypes.POINTER(sz)], ctypes.c_int),
            "ck_init_state": ([vp, vp, sz, vp, u32, u32, u32, u64, u32, vp], ctypes.c_int),
            "ck_turn": ([vp, vp, sz, u32, vp, ctypes.POINTER(TurnResult)], ctypes.c_int),
            "ck_turn_batch": ([vp, vp, vp, u32, vp, vp, vp], ctypes.c_int),
            "ck_tokenizer_load": ([vp, sz, u32, ctypes.POINTER(vp)], ctypes.c_int),
            "ck_tokenizer_free": ([vp], None),
            "ck_encode": ([vp, vp, sz, vp, u32, ctypes.POINTER(u32)], ctypes.c_int),
            "ck_decode": ([vp, u32, vp, u32, vp, sz, ctypes.POINTER(sz)], ctypes.c_int),
            "ck_page_size": ([vp, u32, u32, ctypes.POINTER(sz)], ctypes.c_int),
            "ck_state_to_page": ([vp, vp, vp, sz, vp, sz, vp, sz], ctypes.c_int),
            "ck_state_from_page": ([vp, vp, sz, vp, sz], ctypes.c_int),
            "ck_turn_noalloc": ([vp, vp, sz, vp, ctypes.POINTER(TurnResult)], ctypes.c_int),
            "ck_logits": ([vp, vp, sz, vp, vp], ctypes.c_int),
            "ck_argmax": ([vp, vp, sz, ctypes.POINTER(u32), vp], ctypes.c_int),
            "ck_output_tokens": ([vp, vp, sz, vp, u32, ctypes.POINTER(u32), vp], ctypes.c_int),
            "ck_state_download": ([vp, sz, vp, vp], ctypes.c_int),
            "ck_state_upload": ([vp, vp, sz, vp], ctypes.c_int),
            "ck_matrow": ([vp, sz, vp, u32, u32, vp, vp, vp], ctypes.c_int),
            "ck_host_isqrt": ([u64], u64),
            "ck_host_div_trunc": ([i64, u32], i64),
            "ck_host_probability": ([u64, u64], u64),
            "ck_version": ([], ctypes.c_char_p),
        }
        for name, (args, res) in sig.items():
            f = getattr(L, name)
            f.argtypes = args
            f.restype = res
        _lib = L
    return _lib


def _stream(stream=None):
    import torch
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def _ptr(t) -> ctypes.c_void_p:
    return ctypes.c_void_p(t.data_ptr())


def _host(a: np.ndarray, dtype) -> np.ndarray:
    return np.ascontiguousarray(a, dtype=dtype)


def model_size(artifact: np.ndarray) -> tuple[int, int]:
    art = _host(artifact, np.uint8)
    out = ctypes.c_size_t()
    rc = lib().ck_model_size(art.ctypes.data, art.size, ctypes.byref(out))
    return rc, out.value


class Model:
    """A model in HBM.  ``load`` returns (rc, Model or None)."""

    def __init__(self, handle, mem, config):
        self._h = handle
        self.mem = mem            # the torch tensor holding the device copy
        self.config = config

    @classmethod
    def load(cls, artifact: np.ndarray, stream=None):
        import torch
        art = _host(artifact, np.uint8)
        rc, size = model_size(art)
        if rc:
            return rc, None
        mem = torch.empty(size + 256, dtype=torch.uint8, device="cuda")
        off = (-mem.data_ptr()) % 256
        view = mem[off:off + size]
        h = ctypes.c_void_p()
        rc = lib().ck_load_model(art.ctypes.data, art.size, _ptr(view), size, _stream(stream), ctypes.byref(h))
        if rc:
            return rc, None
        cfg = Config()
        lib().ck_model_config(h, ctypes.byref(cfg))
        return 0, cls(h, mem, {n: getattr(cfg, n) for n, _ in Config._fields_})

    def close(self):
        if self._h:
            lib().ck_free_model(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def set_path(self, path: int) -> int:
        """PATH_AUTO, PATH_STEP (one persistent kernel per position) or PATH_KERNELS."""
        return lib().ck_set_path(self._h, path)

    def set_step_slots(self, max_slots: int) -> int:
        """Cap on the persistent kernel's ring slots (0: as many as fit)."""
        return lib().ck_set_step_slots(self._h, max_slots)

    def set_step_wait_limit(self, polls: int) -> int:
        """Polls of the one-position kernel's barriers before they give up (0: default)."""
        return lib().ck_set_step_wait_limit(self._h, polls)

    def set_step_prefetch(self, kb_per_block: int) -> int:
        """L2 prefetch distance of the persistent kernel, KB per block (0: default)."""
        return lib().ck_set_step_prefetch(self._h, kb_per_block)

    def set_prefill(self, positions: int) -> int:
        """Prompt positions per layer-major prefill chunk (0 or 1: position by position)."""
        return lib().ck_set_prefill(self._h, positions)

    def set_attention_split(self, positions: int) -> int:
        """Positions up to which each block of an attention head scores all of them (0: default)."""
        return lib().ck_set_attention_split(self._h, positions)

    def state_size(self, n_prompt: int, max_tokens: int) -> tuple[int, int]:
        out = ctypes.c_size_t()
        rc = lib().ck_state_size(self._h, n_prompt, max_tokens, ctypes.byref(out))
        return rc, out.value

    def new_state(self, n_prompt: int, max_tokens: int):
        """A zeroed device buffer of the state size (torch allocations are 512-byte aligned)."""
        import torch
        rc, size = self.state_size(n_prompt, max_tokens)
        if rc:
            raise CkError(rc, "ck_state_size")
        return torch.zeros(size, dtype=torch.uint8, device="cuda")

    def init_state(self, state, ids, max_tokens: int, temperature_q16: int = 0, seed: int = 0,
                   flags: int = 0, length: int | None = None, stream=None) -> int:
        ids = _host(np.asarray(ids), np.uint32)
        n = state.numel() if length is None else length
        return lib().ck_init_state(self._h, _ptr(state), n, ids.ctypes.data if ids.size else None,
                                   ids.size, max_tokens, temperature_q16, seed, flags, _stream(stream))

    def turn(self, state, n_positions: int, length: int | None = None, stream=None):
        res = TurnResult()
        n = state.numel() if length is None else length
        rc = lib().ck_turn(self._h, _ptr(state), n, n_positions, _stream(stream), ctypes.byref(res))
        return rc, res.as_dict()

    def turn_batch(self, states, lengths=None, stream=None):
        """One position of each state in one batched pass (ck_turn_batch).
        Returns (rc, [result dict per state], [rc per state])."""
        n = len(states)
        ptrs = (ctypes.c_void_p * max(n, 1))(*[_ptr(t) for t in states])
        lens = (ctypes.c_size_t * max(n, 1))(*[(t.numel() if lengths is None else lengths[i])
                                             for i, t in enumerate(states)])
        res = (TurnResult * max(n, 1))()
        rcs = (ctypes.c_int * max(n, 1))()
        rc = lib().ck_turn_batch(self._h, ptrs, lens, n, _stream(stream), res, rcs)
        return rc, [res[i].as_dict() for i in range(n)], [int(rcs[i]) for i in range(n)]

    def state_to_page(self, tokenizer, host_state, prompt: bytes):
        """This library's state (host bytes) into the page's CURTAST2 state.  Returns (rc, page)."""
        n = ctypes.c_size_t()
        rc = lib().ck_page_size(self._h, len(prompt), int(host_state[20:24].view("<u4")[0]), ctypes.byref(n))
        if rc:
            return rc, None
        page = np.zeros(n.value, dtype=np.uint8)
        p = np.frombuffer(bytes(prompt) or b"\0", dtype=np.uint8)
        hs = np.ascontiguousarray(host_state)
        rc = lib().ck_state_to_page(self._h, tokenizer._h, hs.ctypes.data, hs.size, p.ctypes.data, len(prompt),
                                    page.ctypes.data, page.size)
        return rc, page

    def state_from_page(self, page, n_prompt: int, max_tokens: int):
        """A page state at a position boundary into this library's state (host bytes).
        Returns (rc, state)."""
        rc, n = self.state_size(n_prompt, max_tokens)
        if rc:
            return rc, None
        st = np.zeros(n, dtype=np.uint8)
        pg = np.ascontiguousarray(page)
        rc = lib().ck_state_from_page(self._h, pg.ctypes.data, pg.size, st.ctypes.data, st.size)
        return rc, st

    def turn_noalloc(self, state, stream=None):
        """One position through ck_turn_noalloc (no device allocation, shared scratch)."""
        res = TurnResult()
        rc = lib().ck_turn_noalloc(self._h, _ptr(state), state.numel(), _stream(stream), ctypes.byref(res))
        return rc, res.as_dict()

    def logits(self, state, stream=None):
        out = np.zeros(self.config["vocab"], dtype=np.int64)
        rc = lib().ck_logits(self._h, _ptr(state), state.numel(), out.ctypes.data, _stream(stream))
        return rc, out

    def argmax(self, state, stream=None):
        out = ctypes.c_uint32()
        rc = lib().ck_argmax(self._h, _ptr(state), state.numel(), ctypes.byref(out), _stream(stream))
        return rc, out.value

    def output_tokens(self, state, cap: int | None = None, stream=None):
        cap = self.config["context"] if cap is None else cap
        out = np.zeros(max(cap, 1), dtype=np.uint32)
        n = ctypes.c_uint32()
        rc = lib().ck_output_tokens(self._h, _ptr(state), state.numel(), out.ctypes.data, cap,
                                    ctypes.byref(n), _stream(stream))
        return rc, out[:n.value].tolist()


class Tokenizer:
    """A vocabulary for phases 0 to 2 and token text (host code in the library)."""

    def __init__(self, handle):
        self._h = handle

    @classmethod
    def load(cls, blob: bytes, vocab: int):
        """Returns (rc, Tokenizer or None)."""
        b = np.frombuffer(bytes(blob), dtype=np.uint8)
        h = ctypes.c_void_p()
        rc = lib().ck_tokenizer_load(b.ctypes.data, b.size, vocab, ctypes.byref(h))
        return rc, (cls(h) if rc == 0 else None)

    def __del__(self):
        try:
            if self._h:
                lib().ck_tokenizer_free(self._h)
        except Exception:
            pass

    def encode(self, text: bytes):
        """Returns (rc, ids)."""
        t = np.frombuffer(bytes(text) or b"\0", dtype=np.uint8)
        cap = len(text) + 2
        ids = np.zeros(cap, dtype=np.uint32)
        n = ctypes.c_uint32()
        rc = lib().ck_encode(self._h, t.ctypes.data, len(text), ids.ctypes.data, cap, ctypes.byref(n))
        return rc, (ids[:n.value].copy() if rc == 0 else np.zeros(0, np.uint32))

    def decode(self, ids, prev: int = 0):
        """Returns (rc, text bytes)."""
        a = np.ascontiguousarray(np.asarray(ids, dtype=np.uint32))
        n = ctypes.c_size_t()
        cap = 256 * max(a.size, 1)
        out = np.zeros(cap, dtype=np.uint8)
        rc = lib().ck_decode(self._h, prev, a.ctypes.data if a.size else None, a.size, out.ctypes.data, cap,
                             ctypes.byref(n))
        return rc, out[:n.value].tobytes()


def state_download(state, stream=None) -> np.ndarray:
    host = np.zeros(state.numel(), dtype=np.uint8)
    rc = lib().ck_state_download(_ptr(state), host.size, host.ctypes.data, _stream(stream))
    if rc:
        raise CkError(rc, "ck_state_download")
    return host


def state_upload(state, host: np.ndarray, stream=None) -> None:
    host = _host(host, np.uint8)
    assert host.size == state.numel()
    rc = lib().ck_state_upload(_ptr(state), host.ctypes.data, host.size, _stream(stream))
    if rc:
        raise CkError(rc, "ck_state_upload")


def matrow(W, scale, x, out=None, cols: int | None = None, stream=None):
    """y = matrix row of W (device uint8 [rows][pitch]) and x (device int64); returns (rc, y)."""
    import torch
    rows, pitch = W.shape
    cols = pitch if cols is None else cols
    if out is None:
        out = torch.empty(rows, dtype=torch.int64, device=W.device)
    rc = lib().ck_matrow(_ptr(W), pitch, _ptr(scale), rows, cols, _ptr(x), _ptr(out), _stream(stream))
    return rc, out


def host_isqrt(v: int) -> int:
    return int(lib().ck_host_isqrt(v))


def host_div_trunc(n: int, d: int) -> int:
    return int(lib().ck_host_div_trunc(n, d))


def host_probability(e: int, z: int) -> int:
    """Host build of the attention kernels' floor((e << 24) / z)."""
    return int(lib().ck_host_probability(e, z))


def version() -> str:
    return lib().ck_version().decode()
