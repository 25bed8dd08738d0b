"""Whole-model checks of the CPU oracle: invariants and special cases that hold whatever
the weights are ("The inference core": "The forward pass, in order", "Attention, stage by
stage", "The resumable state", "Core errors")."""
import dataclasses

import numpy as np
import pytest

import oracle
import synth


def _model(spec):
    return oracle.Model(synth.build_artifact(spec))


def _buf(m, st, wl, name, dtype, count):
    lay = m.layout(wl.n_prompt, wl.steps)
    o = lay[name]
    return st[o:o + np.dtype(dtype).itemsize * count].view(dtype)


@pytest.fixture(scope="module")
def tiny_ws():
    wl = synth.WORKLOADS["tiny_ws"]
    return wl, _model(wl.spec)


def test_literal_tiny_config_overflows_the_cache():
    # the tiny workload as written (row scales ~2^24/8) grows the residual past 2^32 in the
    # first layer, so layer 2's key store fails on the second position with error 8
    wl = synth.WORKLOADS["tiny"]
    m = _model(wl.spec)
    rc, st = m.init_state(synth.prompt_ids(wl.spec, wl.n_prompt), wl.steps)
    assert rc == 0
    oracle.events_reset(True)
    rc, res = m.turn(st, 100)
    ev = oracle.events()
    oracle.events_reset(False)
    assert rc == 8 and res["complete"] == 1 and res["work"] == 2
    assert (res["err_position"], res["err_layer"], res["err_phase"]) == (1, 1, 6)
    assert ev["norm_squares"] > 0          # the 64-bit range really was left
    h = oracle.header(st)
    assert h["phase"] == oracle.PHASE_FAILED and h["error"] == 8
    # a failed state cannot take another turn
    assert m.turn(st, 1)[0] == 3


def test_well_scaled_models_stay_in_range(tiny_ws):
    wl, m = tiny_ws
    rc, st = m.init_state(synth.prompt_ids(wl.spec, wl.n_prompt), wl.steps)
    oracle.events_reset(True)
    rc, res = m.turn(st, 1000)
    ev = oracle.events()
    oracle.events_reset(False)
    assert rc == 0 and res["complete"] and res["generated"] == wl.steps
    assert res["work"] == wl.n_prompt + wl.steps - 1
    assert all(v == 0 for v in ev.values()), ev


@pytest.mark.parametrize("name", ["tiny_ws", "gqa"])
def test_position_zero_attention_returns_the_value_row(name):
    # with one position the probability is exactly 2^24, so each head's output equals its
    # key/value head's cached value row; the value head of head h is h / (heads / kv_heads)
    wl = synth.WORKLOADS[name]
    spec = wl.spec
    m = _model(spec)
    rc, st = m.init_state(synth.prompt_ids(spec, wl.n_prompt), wl.steps)
    rc, res = m.turn(st, 1)
    assert rc == 0 and res["work"] == 1
    cache = wl.n_prompt + wl.steps - 1
    o = _buf(m, st, wl, "o", "<i8", spec.dim)
    hd, group = spec.head_dim, spec.heads // spec.kv_heads
    # the cache is head-major: [layer][kv head][position][head element]
    V = _buf(m, st, wl, "v", "<i4", spec.layers * cache * spec.kv_dim).reshape(
        spec.layers, spec.kv_heads, cache, hd)
    for h in range(spec.heads):
        kvh = h // group
        assert o[h * hd:(h + 1) * hd].tolist() == V[-1, kvh, 0].astype(np.int64).tolist()


def test_turn_split_invariance(tiny_ws):
    wl, m = tiny_ws
    ids = synth.prompt_ids(wl.spec, wl.n_prompt)
    _, a = m.init_state(ids, wl.steps)
    m.turn(a, 1000)
    _, b = m.init_state(ids, wl.steps)
    for n in (1, 2, 3, 5, 1000):
        if oracle.header(b)["phase"] != oracle.PHASE_RUNNING:
            break
        m.turn(b, n)
    ha, hb = oracle.header(a), oracle.header(b)
    assert hb["turns"] > ha["turns"]
    a[56:64] = 0
    b[56:64] = 0                            # only the turn counter may differ
    assert np.array_equal(a, b)


def test_stop_tokens_end_the_run(tiny_ws):
    wl, m = tiny_ws
    ids = synth.prompt_ids(wl.spec, wl.n_prompt)
    _, full = m.init_state(ids, wl.steps)
    m.turn(full, 1000)
    toks = _buf(m, full, wl, "out", "<u4", wl.steps).tolist()
    first = next(i for i, t in enumerate(toks) if t in (1, 2))   # this seed emits one
    _, st = m.init_state(ids, wl.steps, flags=oracle.FLAG_STOP_TOKENS)
    rc, res = m.turn(st, 1000)
    assert rc == 0 and res["complete"] and res["generated"] == first + 1
    assert res["token"] == toks[first]
    assert oracle.header(st)["phase"] == oracle.PHASE_DONE
    assert _buf(m, st, wl, "out", "<u4", wl.steps).tolist()[:first + 1] == toks[:first + 1]


def test_init_state_errors(tiny_ws):
    wl, m = tiny_ws
    ids = synth.prompt_ids(wl.spec, 4)
    ctx = wl.spec.context
    assert m.init_state(ids, 0)[0] == 6                       # max tokens zero
    assert m.init_state(ids, ctx + 1)[0] == 6                 # above the context
    assert m.init_state(np.array([wl.spec.vocab], np.uint32), 2)[0] == 6   # id out of range
    assert m.init_state(np.array([], np.uint32), 2)[0] == 6   # no prompt id
    assert m.init_state(ids, 2, temperature_q16=16 * 2**16 + 1)[0] == 6
    assert m.init_state(ids, 2, temperature_q16=16 * 2**16)[0] == 0   # 16 is allowed
    assert m.init_state(ids, ctx - 2)[0] == 7                 # 4 + (ctx-2) - 1 > ctx
    assert m.init_state(ids, ctx - 3)[0] == 0                 # exactly the context
    n = m.state_size(4, 5)
    assert m.init_state(ids, 5, length=n + 8)[0] == 4
    assert m.init_state(ids, 5, length=n - 8)[0] == 4


def test_turn_rejects_foreign_states(tiny_ws):
    wl, m = tiny_ws
    ids = synth.prompt_ids(wl.spec, 4)
    _, st = m.init_state(ids, 5)
    bad = st.copy()
    bad[0] ^= 1
    assert m.turn(bad, 1)[0] == 3                             # tag
    bad = st.copy()
    bad[80] ^= 1
    assert m.turn(bad, 1)[0] == 3                             # configuration echo
    bad = st.copy()
    bad[oracle.H_POSITION] = 8                                # cursor past the cache
    assert m.turn(bad, 1)[0] == 3


def test_artifact_errors():
    art = synth.build_artifact(synth.TINY_WS)
    bad = art.copy()
    bad[0] = ord("X")
    with pytest.raises(ValueError, match="error 2"):
        oracle.Model(bad)
    with pytest.raises(ValueError, match="error 2"):
        oracle.Model(art[:-64].copy())                        # truncated
    bad = art.copy()
    bad[8:12] = 0                                             # dim zero
    with pytest.raises(ValueError, match="error 1"):
        oracle.Model(bad)


def test_tied_classifier_reads_the_embedding():
    # untying with a classifier that is a copy of the embedding gives the same run
    spec = synth.GQA_TIED
    wl = synth.WORKLOADS["gqa_tied"]
    tied = synth.build_artifact(spec)
    untied_spec = dataclasses.replace(spec, tied=False)
    untied = synth.build_artifact(untied_spec)
    synth.artifact_tensor(untied, synth.T_CLS)[...] = synth.artifact_tensor(tied, synth.T_EMBED)
    synth.artifact_tensor(untied, synth.T_CLS_SCALE)[...] = synth.artifact_tensor(tied, synth.T_EMBED_SCALE)
    outs = []
    for art in (tied, untied):
        m = oracle.Model(art)
        rc, st = m.init_state(synth.prompt_ids(spec, wl.n_prompt), wl.steps)
        rc, res = m.turn(st, 1000)
        assert rc == 0
        outs.append(_buf(m, st, wl, "out", "<u4", wl.steps).tolist())
    assert outs[0] == outs[1]


def test_sampled_run_advances_the_generator_once_per_token(tiny_ws):
    """"Sampling": above temperature zero each generated token draws once from the run's
    generator, seeded by the run's seed (a zero seed from the page's constant), and the
    header keeps the last sum of exponentials and draw, with draw < sum."""
    wl, m = tiny_ws
    ids = synth.prompt_ids(wl.spec, wl.n_prompt)
    f_zero = 0x9E3779B97F4A7C15
    for seed, temp in ((0, 1 << 16), (12345, 3 << 15), (2**64 - 1, 16 << 16)):
        rc, st = m.init_state(ids, wl.steps, temperature_q16=temp, seed=seed)
        assert rc == 0
        h = oracle.header(st)
        assert h["generator"] == (seed or f_zero) and h["temperature"] == temp
        state = seed or f_zero
        for pos in range(wl.n_prompt + wl.steps - 1):
            rc, res = m.turn(st, 1)
            assert rc == 0
            h = oracle.header(st)
            if pos + 1 >= wl.n_prompt:
                tok = int(_buf(m, st, wl, "out", "<u4", wl.steps)[h["generated"] - 1])
                lg = _buf(m, st, wl, "logits", "<i8", wl.spec.vocab)
                r = oracle.sample(lg, temp, synth.exp_table(), state)   # from the state before
                state = oracle.xorshift_next(state)[0]
                assert r["token"] == tok and r["state"] == state
                assert (r["sum"], r["draw"]) == (h["exp_sum"], h["draw"])
                assert 0 <= h["draw"] < h["exp_sum"]
                assert h["exp_sum"] >= 1 << 30                # the largest logit adds EXP[0]
                assert h["max_logit"] == int(lg.max())
            else:
                assert h["draw"] == 0 and h["exp_sum"] == 0
            assert h["generator"] == state
        assert h["phase"] == oracle.PHASE_DONE


def test_high_temperature_changes_the_tokens_and_zero_does_not_draw(tiny_ws):
    wl, m = tiny_ws
    ids = synth.prompt_ids(wl.spec, wl.n_prompt)
    _, greedy = m.init_state(ids, wl.steps)
    m.turn(greedy, 1000)
    g = _buf(m, greedy, wl, "out", "<u4", wl.steps).tolist()
    h = oracle.header(greedy)
    assert h["generator"] == 0x9E3779B97F4A7C15 and h["exp_sum"] == 0   # never advanced
    _, hot = m.init_state(ids, wl.steps, temperature_q16=16 << 16, seed=7)
    m.turn(hot, 1000)
    assert _buf(m, hot, wl, "out", "<u4", wl.steps).tolist() != g


# ---------------------------------------------------------------- the page's state (CURTAST2)

def _page_case(temp=0):
    wl = synth.WORKLOADS["gqa"]
    spec = wl.spec
    m = _model(spec)
    blob = synth.tokenizer_blob(spec.vocab, spec.seed)
    v = oracle.Vocab(blob, spec.vocab)
    text = synth.prompt_text(12, spec.seed, 1, blob)
    return spec, m, v, text


def test_page_sizes_agree_with_the_printed_sizes_rule():
    spec, m, v, text = _page_case()
    for pb, mt in ((16, 12), (0, 30), (100, 7)):
        assert oracle.page_layout(m, pb, mt)["size"] == oracle.page_state_size(spec.config(), pb, mt)


def test_page_run_stops_anywhere_and_matches_the_ids_run():
    """The page state run step by step with stops every k steps (mid-layer and mid-attention
    included) ends in the same bytes as one uninterrupted turn, and its tokens, activations,
    logits and cache equal those of the ids-mode run of the same prompt ids."""
    spec, m, v, text = _page_case()
    steps = 9
    rc, ref = oracle.page_new(m, text, steps, 3 << 15, 11)
    assert rc == 0
    rc, n = oracle.page_turn(m, v, ref, 10**9)
    assert rc == 0 and oracle.page_header(ref)["phase"] == 20
    for k in (1, 5, 23):
        rc, st = oracle.page_new(m, text, steps, 3 << 15, 11)
        turns = 0
        while oracle.page_header(st)["phase"] != 20:
            rc, ran = oracle.page_turn(m, v, st, k)
            assert rc == 0 and ran >= 1
            turns += 1
        assert turns > 1
        a, b = ref.copy(), st.copy()
        a[80:88] = 0
        b[80:88] = 0                                           # the turn counters differ
        assert np.array_equal(a, b), k
    # the ids-mode oracle on the page's prompt tokens
    pl = oracle.page_layout(m, len(text), steps)
    h = oracle.page_header(ref)
    ids = ref[pl["ptok"]:pl["ptok"] + 4 * h["prompt_tokens"]].view("<u4")
    assert ids.tolist() == v.encode(text)[1]
    rc, so = m.init_state(ids, steps, 3 << 15, 11)
    rco, _ = m.turn(so, 10**6)
    assert rco == 0
    lay = m.layout(len(ids), steps)
    assert ref[pl["out"]:pl["out"] + 4 * steps].tobytes() == so[lay["out"]:lay["out"] + 4 * steps].tobytes()
    for name in ("x", "logits"):
        nb = 8 * (spec.dim if name == "x" else spec.vocab)
        assert ref[pl[name]:pl[name] + nb].tobytes() == so[lay[name]:lay[name] + nb].tobytes(), name
    # caches: the page keeps [layer][position][kv], the ids state [layer][kv head][position][head]
    cache_o = len(ids) + steps - 1
    hd, kvh = spec.head_dim, spec.kv_heads
    for name in ("k", "v"):
        page = ref[pl[name]:pl[name] + 4 * spec.layers * pl["cache"] * spec.kv_dim].view("<i4").reshape(
            spec.layers, pl["cache"], spec.kv_dim)[:, :cache_o]
        mine = so[lay[name]:lay[name] + 4 * spec.layers * cache_o * spec.kv_dim].view("<i4").reshape(
            spec.layers, kvh, cache_o, hd).transpose(0, 2, 1, 3).reshape(spec.layers, cache_o, spec.kv_dim)
        assert np.array_equal(page, mine), name
    text_out = ref[pl["text"]:pl["text"] + h["text_bytes"]].tobytes()
    assert text_out == v.decode(ref[pl["out"]:pl["out"] + 4 * steps].view("<u4").tolist(), prev=int(ids[-1]))
