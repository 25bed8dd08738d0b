"""ck_turn_noalloc: the one-position entry point for callers that cannot allocate device
memory while running (a server whose device memory is split into fixed arenas up front, a
host framework that owns every allocation).  It must give exactly the bits of ck_turn on
the persistent kernel and of the CPU oracle.  Two calls in a row cover a prompt position
(it ends with the last residual) and a generating position (classifier and maximum pass),
and the second call shows that the shared scratch array is cleared between calls.

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
    """Two calls in a row against ck_turn on the persistent kernel and against the oracle,
    state buffer by state buffer; the device's free memory is the same before and after the
    two calls (nothing allocated, nothing freed)."""
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
    orc = oracle.Model(art)
    ids = synth.prompt_ids(spec, n_prompt)
    ref = model.new_state(n_prompt, max_tokens)
    got = model.new_state(n_prompt, max_tokens)
    warm = model.new_state(n_prompt, max_tokens)
    assert model.init_state(ref, ids, max_tokens) == 0
    assert model.init_state(got, ids, max_tokens) == 0
    assert model.init_state(warm, ids, max_tokens) == 0
    rc, so = orc.init_state(ids, max_tokens)
    assert rc == 0
    lay = orc.layout(n_prompt, max_tokens)
    # a first call on another state does the once-per-device set-up before the measurement
    assert model.turn_noalloc(warm)[0] == 0
    torch.cuda.synchronize()
    free_before = torch.cuda.mem_get_info()[0]
    results = []
    for call in range(2):
        rc_got, res_got = model.turn_noalloc(got)
        results.append((rc_got, res_got, ck.state_download(got)))
    torch.cuda.synchronize()
    free_after = torch.cuda.mem_get_info()[0]
    assert free_after == free_before, (free_before, free_after)
    for call, (rc_got, res_got, host_got) in enumerate(results):
        rc_ref, res_ref = model.turn(ref, 1)
        rc_orc, res_orc = orc.turn(so, 1)
        assert rc_ref == rc_got == rc_orc == 0, (call, rc_ref, rc_got, rc_orc)
        assert res_ref == res_got == res_orc, (call, res_ref, res_got, res_orc)
        a = _specified_buffers(lay, ck.state_download(ref), n_prompt, max_tokens, spec.dim, spec.vocab)
        b = _specified_buffers(lay, host_got, n_prompt, max_tokens, spec.dim, spec.vocab)
        c = _specified_buffers(lay, so, n_prompt, max_tokens, spec.dim, spec.vocab)
        for pa, pb, pc in zip(a, b, c):
            assert np.array_equal(pa, pb), f"call {call}: differs from ck_turn"
            assert np.array_equal(pb, pc), f"call {call}: differs from the oracle"
    assert res_got["generated"] == 1
    torch.cuda.synchronize()
