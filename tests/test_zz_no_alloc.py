"""ck_turn_noalloc: the one-position entry point for callers that cannot allocate device
memory while running (a server whose device memory is split into fixed arenas up front, a
host framework that owns every allocation).  It must give exactly the bits of ck_turn on
the persistent kernel.  Two calls in a row cover a prompt position (it ends with the last
residual) and a generating position (classifier and maximum pass), and the second call
shows that the shared scratch array is cleared between calls.

Collected last on purpose: if it fails, a run that stops at the first failure has already
run every other test."""
import numpy as np
import pytest

import oracle
import synth

pytestmark = pytest.mark.gpu


def _specified_buffers(lay, state, n_prompt, max_tokens, dim, vocab):
    """The state fields with specified contents (the working vectors are scratch)."""
    parts = [state[:128]]
    for name, nbytes in (("prompt", 4 * n_prompt), ("out", 4 * max_tokens), ("x", 8 * dim),
                         ("logits", 8 * vocab)):
        parts.append(state[lay[name]:lay[name] + nbytes])
    parts.append(state[lay["k"]:lay["size"]])
    return parts


def test_noalloc_turn_matches_ck_turn_on_two_calls():
    import torch
    import fixed_point_int8_gb300 as ck
    from fixed_point_int8_gb300 import build
    build.build()
    spec = synth.GQA
    n_prompt, max_tokens = 2, 6
    art = synth.build_artifact(spec)
    rc, model = ck.Model.load(art)
    assert rc == 0
    assert model.set_path(ck.PATH_STEP) == 0
    ids = synth.prompt_ids(spec, n_prompt)
    ref = model.new_state(n_prompt, max_tokens)
    got = model.new_state(n_prompt, max_tokens)
    assert model.init_state(ref, ids, max_tokens) == 0
    assert model.init_state(got, ids, max_tokens) == 0
    lay = oracle.Model(art).layout(n_prompt, max_tokens)
    for call in range(2):
        rc_ref, res_ref = model.turn(ref, 1)
        rc_got, res_got = model.turn_noalloc(got)
        assert rc_ref == rc_got == 0, (call, rc_ref, rc_got)
        assert res_ref == res_got, (call, res_ref, res_got)
        a = _specified_buffers(lay, ck.state_download(ref), n_prompt, max_tokens, spec.dim, spec.vocab)
        b = _specified_buffers(lay, ck.state_download(got), n_prompt, max_tokens, spec.dim, spec.vocab)
        for pa, pb in zip(a, b):
            assert np.array_equal(pa, pb), f"call {call}: state differs"
    assert res_got["generated"] == 1
    torch.cuda.synchronize()
