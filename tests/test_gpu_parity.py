"""GPU parity: the CUDA path through the C ABI against the CPU oracle, element by element,
bit-exact (integer work, tolerance 0)."""
import dataclasses

import numpy as np
import pytest

import oracle
import synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ck():
    import torch
    import fixed_point_int8_gb300 as ck
    from fixed_point_int8_gb300 import build
    build.build()
    torch.cuda.init()
    return ck


# ---------------------------------------------------------------- helpers

PATHS = {"step": 1, "kernels": 2}   # one persistent kernel per position / one kernel per phase


class Pair:
    """The same artifact loaded into the oracle and into the GPU library."""

    def __init__(self, ck, spec, path="step"):
        self.spec = spec
        self.path = path
        self.art = synth.build_artifact(spec)
        self.orc = oracle.Model(self.art)
        rc, self.gpu = ck.Model.load(self.art)
        assert rc == 0, rc
        assert self.gpu.set_path(PATHS[path]) == 0

    def init(self, ck, ids, max_tokens, flags=0, temperature_q16=0, seed=0):
        rc, so = self.orc.init_state(ids, max_tokens, temperature_q16, seed, flags=flags)
        assert rc == 0
        sg = self.gpu.new_state(len(ids), max_tokens)
        assert self.gpu.init_state(sg, ids, max_tokens, temperature_q16, seed, flags=flags) == 0
        return so, sg


# Working vectors (scratch in the state format) that a path leaves with the oracle's
# contents after a position it runs alone: the phase kernels write the last layer's rotated
# queries, head outputs, down-row output and SiLU output where the oracle does; the
# persistent kernel writes only the queries there.
VECTORS = {"kernels": ("q", "o", "y", "h"), "step": ("q",)}


def compare_states(orc_model, so, sg_host, n_prompt, max_tokens, what="", turns=True, vectors=()):
    """Every specified field and buffer of two states (the working vectors are scratch,
    except those named in `vectors`).  turns=False skips the turn counter, for runs split
    into different numbers of turns."""
    lay = orc_model.layout(n_prompt, max_tokens)
    assert so.size == sg_host.size == lay["size"]
    ho, hg = oracle.header(so), oracle.header(sg_host)
    if not turns:
        ho.pop("turns"), hg.pop("turns")
    assert ho == hg, (what, ho, hg)
    assert np.array_equal(so[:8], sg_host[:8])
    assert np.array_equal(so[80:108], sg_host[80:108]), what
    d, v = orc_model.config[0], orc_model.config[5]
    for name, nbytes in (("prompt", 4 * n_prompt), ("out", 4 * max_tokens), ("x", 8 * d),
                         ("logits", 8 * v)):
        o = lay[name]
        a, b = so[o:o + nbytes], sg_host[o:o + nbytes]
        if not np.array_equal(a, b):
            bad = np.flatnonzero(a != b)
            raise AssertionError(f"{what}: buffer {name} differs at byte {bad[:8]}")
    hidden = orc_model.config[1]
    for name in vectors:
        o, nbytes = lay[name], 8 * (hidden if name == "h" else d)
        a, b = so[o:o + nbytes], sg_host[o:o + nbytes]
        if not np.array_equal(a, b):
            bad = np.flatnonzero(a != b)
            raise AssertionError(f"{what}: working vector {name} differs at byte {bad[:8]}")
    for name in ("k", "v"):
        o, end = lay[name], (lay["v"] if name == "k" else lay["size"])
        a, b = so[o:end], sg_host[o:end]
        if not np.array_equal(a, b):
            bad = np.flatnonzero(a != b)
            raise AssertionError(f"{what}: cache {name} differs at byte offset {bad[:8]}")


# ---------------------------------------------------------------- matrix row

# (rows, cols, pitch).  Past 38,912 rows a CTA finishes its share in several 256-row chunks
# (80,001: odd, three chunks a CTA); a pitch that is not a multiple of 512 leaves a partial
# last slice.
MATROW_CASES = [(1, 1, 16), (3, 15, 16), (5, 17, 32), (7, 172, 176), (64, 64, 64), (130, 300, 304),
                (1001, 1000, 1008), (257, 4096, 4096), (64, 11008, 11008), (33, 16384, 16384),
                (80001, 48, 64), (40000, 130, 144)]


def _x_for_limbs(L, cols, seed):
    rng = np.random.default_rng(seed)
    if L == 8:
        x = rng.integers(-2**63, 2**63 - 1, cols, dtype=np.int64)
        x[:4] = [-2**63, 2**63 - 1, -1, 0][: min(4, cols)]
        return x
    lim = 2**(8 * L - 1)
    x = rng.integers(-lim, lim, cols, dtype=np.int64)     # [-lim, lim - 1]: exactly L limbs
    x[0] = -lim
    if cols > 1:
        x[1] = lim - 1
    return x


@pytest.mark.parametrize("rows,cols,pitch", MATROW_CASES)
def test_matrow_every_limb_count(ck, rows, cols, pitch):
    import torch
    W, s, _ = synth.matrow_case(rows, cols, pitch=pitch)
    W[0, :cols] = 255
    if rows > 1:
        W[1, :cols] = 0
    Wd = torch.from_numpy(W).cuda()
    sd = torch.from_numpy(s.view(np.int32)).cuda()
    for L in range(1, 9):
        x = _x_for_limbs(L, cols, seed=rows * 31 + L)
        want = oracle.matrow(W, s, x, cols=cols)
        rc, y = ck.matrow(Wd, sd, torch.from_numpy(x).cuda(), cols=cols)
        assert rc == 0
        got = y.cpu().numpy()
        assert np.array_equal(got, want), (rows, cols, L, np.flatnonzero(got != want)[:5])


def test_matrow_zero_vector_and_extreme_scales(ck):
    import torch
    W, s, x = synth.matrow_case(40, 48)
    s[:4] = [0, 1, 2**32 - 1, 2**31]
    for vec in (np.zeros(48, np.int64), x):
        want = oracle.matrow(W, s, vec)
        rc, y = ck.matrow(torch.from_numpy(W).cuda(), torch.from_numpy(s.view(np.int32)).cuda(),
                          torch.from_numpy(vec).cuda())
        assert rc == 0 and np.array_equal(y.cpu().numpy(), want)


@pytest.mark.parametrize("rows,cols", synth.MATROW_SHAPES)
def test_matrow_sweep_full_size(ck, rows, cols):
    """The matrix-row sweep at its full sizes, every output row against the oracle."""
    import torch
    W, s, x = synth.matrow_case(rows, cols)
    want = oracle.matrow(W, s, x)
    rc, y = ck.matrow(torch.from_numpy(W).cuda(), torch.from_numpy(s.view(np.int32)).cuda(),
                      torch.from_numpy(x).cuda())
    assert rc == 0
    assert np.array_equal(y.cpu().numpy(), want)


def test_matrow_rejects_bad_arguments(ck):
    import torch
    W = torch.zeros((4, 32), dtype=torch.uint8, device="cuda")
    s = torch.zeros(4, dtype=torch.int32, device="cuda")
    x = torch.zeros(32, dtype=torch.int64, device="cuda")
    assert ck.matrow(W, s, x, cols=33)[0] == 10                    # cols beyond the pitch
    W2 = torch.zeros((4, 24), dtype=torch.uint8, device="cuda")
    assert ck.matrow(W2, s, x, cols=24)[0] == 10                   # pitch not a multiple of 16
    assert ck.matrow(W[:, 1:17], s, x, cols=16)[0] == 10           # misaligned matrix


# ---------------------------------------------------------------- whole model

MODELS = {
    "tiny_ws": synth.WORKLOADS["tiny_ws"],
    "gqa": synth.WORKLOADS["gqa"],
    "gqa_tied": synth.WORKLOADS["gqa_tied"],
}


@pytest.mark.parametrize("slots", [2, 3, 5])
def test_step_kernel_with_a_small_ring(ck, slots):
    """The persistent kernel with fewer ring slots than consumer warps: every slot is reused
    many times within each phase, on a small model, against the oracle position by position."""
    wl = MODELS["gqa"]
    P = Pair(ck, wl.spec, "step")
    assert P.gpu.set_step_slots(slots) == 0
    ids = synth.prompt_ids(wl.spec, wl.n_prompt)
    so, sg = P.init(ck, ids, wl.steps)
    for pos in range(8):
        rco, reso = P.orc.turn(so, 1)
        rcg, resg = P.gpu.turn(sg, 1)
        assert rco == rcg == 0 and reso == resg, (pos, rcg, resg)
        compare_states(P.orc, so, ck.state_download(sg), wl.n_prompt, wl.steps, f"slots {slots} pos {pos}")
    rco, _ = P.orc.turn(so, 10_000)
    rcg, _ = P.gpu.turn(sg, 10_000)
    assert rco == rcg == 0
    compare_states(P.orc, so, ck.state_download(sg), wl.n_prompt, wl.steps, f"slots {slots}", turns=False)
    assert P.gpu.set_step_slots(1) == 10
    assert P.gpu.set_step_slots(9) == 10


@pytest.mark.parametrize("name,split", [("gqa", 1), ("gqa", 3), ("tiny_ws", 1), ("gqa_tied", 2)])
def test_step_kernel_with_split_attention_scoring(ck, name, split):
    """The persistent kernel with each head's scoring split over its blocks beyond `split`
    positions (maxima and sums exchanged between the blocks), every position against the
    oracle."""
    wl = MODELS[name]
    P = Pair(ck, wl.spec, "step")
    assert P.gpu.set_attention_split(split) == 0
    ids = synth.prompt_ids(wl.spec, wl.n_prompt)
    so, sg = P.init(ck, ids, wl.steps)
    for pos in range(wl.n_prompt + wl.steps - 1):
        rco, reso = P.orc.turn(so, 1)
        rcg, resg = P.gpu.turn(sg, 1)
        assert rco == rcg == 0 and reso == resg, (pos, rcg, resg)
        compare_states(P.orc, so, ck.state_download(sg), wl.n_prompt, wl.steps, f"split {split} pos {pos}")


def test_step_kernel_with_l2_prefetch(ck):
    """The persistent kernel with its producer prefetching weights into L2 ahead of a small
    ring: every position against the oracle; out-of-range settings are rejected."""
    wl = MODELS["gqa"]
    P = Pair(ck, wl.spec, "step")
    assert P.gpu.set_step_prefetch(64) == 0
    assert P.gpu.set_step_slots(3) == 0
    ids = synth.prompt_ids(wl.spec, wl.n_prompt)
    so, sg = P.init(ck, ids, wl.steps)
    for pos in range(wl.n_prompt + wl.steps - 1):
        rco, reso = P.orc.turn(so, 1)
        rcg, resg = P.gpu.turn(sg, 1)
        assert rco == rcg == 0 and reso == resg, (pos, rcg, resg)
        compare_states(P.orc, so, ck.state_download(sg), wl.n_prompt, wl.steps, f"prefetch pos {pos}")
    assert P.gpu.set_step_prefetch(5000) == 10


def test_step_kernel_barrier_timeout_fails_the_state_with_error_9(ck):
    """The persistent kernel's timeout path, driven without a fault: with its barrier waits
    cut to one poll, the first grid barrier gives up in the blocks that arrive before the
    last; every block leaves (each producer first waits for its own copies in flight), the
    turn returns 9 and the state is failed with error 9, the stream is idle afterwards, and
    the allocation-free entry fails the same way.  Back at the default limit, a fresh state
    on the same model runs bit-exact against the oracle."""
    import torch
    wl = MODELS["gqa"]
    P = Pair(ck, wl.spec, "step")
    ids = synth.prompt_ids(wl.spec, wl.n_prompt)
    assert P.gpu.set_step_wait_limit(1) == 0
    for entry in ("turn", "noalloc"):
        so, sg = P.init(ck, ids, wl.steps)
        rc, res = P.gpu.turn(sg, 1) if entry == "turn" else P.gpu.turn_noalloc(sg)
        torch.cuda.current_stream().synchronize()
        assert rc == 9 and res["complete"] == 1, (entry, rc, res)
        h = oracle.header(ck.state_download(sg))
        assert h["phase"] == oracle.PHASE_FAILED and h["error"] == 9 and h["position"] == 0, (entry, h)
        assert P.gpu.turn(sg, 1)[0] == 3                       # a failed state is refused
    assert P.gpu.set_step_wait_limit(0) == 0
    so, sg = P.init(ck, ids, wl.steps)
    for pos in range(wl.n_prompt + 2):
        rco, reso = P.orc.turn(so, 1)
        rcg, resg = P.gpu.turn(sg, 1)
        assert rco == rcg == 0 and reso == resg, (pos, rcg, resg)
        compare_states(P.orc, so, ck.state_download(sg), wl.n_prompt, wl.steps, f"after timeout pos {pos}",
                       vectors=VECTORS["step"])


@pytest.fixture(scope="module", params=list(PATHS))
def pairs(ck, request):
    return {name: Pair(ck, wl.spec, request.param) for name, wl in MODELS.items()}


@pytest.mark.parametrize("name", list(MODELS))
def test_every_position_matches_the_oracle(ck, pairs, name):
    wl = MODELS[name]
    P = pairs[name]
    ids = synth.prompt_ids(wl.spec, wl.n_prompt)
    so, sg = P.init(ck, ids, wl.steps)
    compare_states(P.orc, so, ck.state_download(sg), wl.n_prompt, wl.steps, "after init")
    for pos in range(wl.n_prompt + wl.steps - 1):
        rco, reso = P.orc.turn(so, 1)
        rcg, resg = P.gpu.turn(sg, 1)
        assert rco == rcg == 0
        assert reso == resg, (pos, reso, resg)
        compare_states(P.orc, so, ck.state_download(sg), wl.n_prompt, wl.steps, f"position {pos}",
                       vectors=VECTORS[P.path])
    assert oracle.header(so)["phase"] == oracle.PHASE_DONE
    rc, toks = P.gpu.output_tokens(sg)
    assert rc == 0 and len(toks) == wl.steps


SAMPLING = [(1 << 16, 0), (16 << 16, 12345), (3 << 14, 2**64 - 1), (1, 99)]


@pytest.mark.parametrize("temp,seed", SAMPLING)
def test_sampled_positions_match_the_oracle(ck, pairs, temp, seed):
    """Phase 19 above temperature zero (sum pass, draw pass, the generator state, sum and
    draw in the header): every position of two models against the oracle."""
    for name in ("gqa", "tiny_ws"):
        wl = MODELS[name]
        P = pairs[name]
        ids = synth.prompt_ids(wl.spec, wl.n_prompt)
        so, sg = P.init(ck, ids, wl.steps, temperature_q16=temp, seed=seed)
        for pos in range(wl.n_prompt + wl.steps - 1):
            rco, reso = P.orc.turn(so, 1)
            rcg, resg = P.gpu.turn(sg, 1)
            assert rco == rcg == 0 and reso == resg, (name, pos, reso, resg)
            compare_states(P.orc, so, ck.state_download(sg), wl.n_prompt, wl.steps,
                           f"{name} temperature {temp} position {pos}", vectors=VECTORS[P.path])
        h = oracle.header(so)
        assert h["phase"] == oracle.PHASE_DONE and h["exp_sum"] >= 1 << 30


WIDE_VOCAB = synth.ModelSpec("wide_vocab", 64, 172, 2, 4, 4, 70001, 64, scale_rule="well", tied=False,
                             seed=0x5EED0031)


@pytest.mark.parametrize("path", list(PATHS))
def test_sampling_over_a_wide_vocabulary(ck, path):
    """A vocabulary of 70,001 entries: the sampler's groups hold several 32-entry chunks
    and the last chunk is ragged; both temperatures against the oracle at every position."""
    P = Pair(ck, WIDE_VOCAB, path)
    ids = synth.prompt_ids(WIDE_VOCAB, 6)
    for temp, seed in ((16 << 16, 5), (1 << 16, 0), (0, 0)):
        so, sg = P.init(ck, ids, 10, temperature_q16=temp, seed=seed)
        for pos in range(15):
            rco, reso = P.orc.turn(so, 1)
            rcg, resg = P.gpu.turn(sg, 1)
            assert rco == rcg == 0 and reso == resg, (temp, pos, reso, resg)
            compare_states(P.orc, so, ck.state_download(sg), 6, 10, f"wide vocab {temp} {pos}")


def test_many_positions_in_one_turn(ck, pairs):
    wl = MODELS["gqa"]
    P = pairs["gqa"]
    ids = synth.prompt_ids(wl.spec, wl.n_prompt)
    so, sg = P.init(ck, ids, wl.steps)
    rco, reso = P.orc.turn(so, 10_000)
    splits = [1, 7, 3, 30, 10_000]
    for n in splits:
        rc, res = P.gpu.turn(sg, n)
        assert rc == 0
        if res["complete"]:
            break
    host = ck.state_download(sg)
    # the turn counter differs (one turn against several); everything else is identical
    compare_states(P.orc, so, host, wl.n_prompt, wl.steps, "split turns", turns=False)
    assert P.gpu.turn(sg, 1)[0] == 3                               # complete: InvalidState


@pytest.mark.parametrize("path", list(PATHS))
def test_literal_tiny_workload_fails_like_the_oracle(ck, path):
    wl = synth.WORKLOADS["tiny"]
    P = Pair(ck, wl.spec, path)
    ids = synth.prompt_ids(wl.spec, wl.n_prompt)
    so, sg = P.init(ck, ids, wl.steps)
    rco, reso = P.orc.turn(so, 100)
    rcg, resg = P.gpu.turn(sg, 100)
    assert rco == rcg == 8
    assert reso == resg
    ho, hg = oracle.header(so), oracle.header(ck.state_download(sg))
    for k in ("phase", "error", "err_key", "position", "generated"):
        assert ho[k] == hg[k], k
    assert P.gpu.turn(sg, 1)[0] == 3


def test_stop_tokens(ck, pairs):
    wl = MODELS["tiny_ws"]
    P = pairs["tiny_ws"]
    ids = synth.prompt_ids(wl.spec, wl.n_prompt)
    so, sg = P.init(ck, ids, wl.steps, flags=ck.CK_FLAG_STOP_TOKENS)
    rco, reso = P.orc.turn(so, 1000)
    rcg, resg = P.gpu.turn(sg, 1000)
    assert rco == rcg == 0 and reso == resg and resg["complete"]
    assert resg["generated"] < wl.steps                  # this seed emits a stop token early
    compare_states(P.orc, so, ck.state_download(sg), wl.n_prompt, wl.steps, "stop tokens")


def test_init_state_errors_match_the_oracle(ck, pairs):
    P = pairs["tiny_ws"]
    spec = P.spec
    ids = synth.prompt_ids(spec, 4)
    ctx = spec.context
    import torch
    big = torch.zeros(1 << 20, dtype=torch.uint8, device="cuda")
    cases = [(ids, 0, 0), (ids, ctx + 1, 0), (np.array([spec.vocab], np.uint32), 2, 0),
             (ids, 2, 16 * 2**16 + 1), (ids, ctx - 2, 0)]
    for i, mt, temp in cases:
        rco = P.orc.init_state(i, mt, temperature_q16=temp)[0]
        rcg = P.gpu.init_state(big, i, mt, temperature_q16=temp)
        assert rco == rcg != 0, (mt, temp, rco, rcg)
    rc, n = P.gpu.state_size(4, 5)
    assert rc == 0
    assert P.gpu.init_state(big, ids, 5, length=n + 8) == 4
    assert P.gpu.init_state(big[8:], ids, 5, length=n) == 3          # misaligned


def test_turn_rejects_foreign_states(ck, pairs):
    P = pairs["tiny_ws"]
    ids = synth.prompt_ids(P.spec, 4)
    sg = P.gpu.new_state(4, 5)
    assert P.gpu.init_state(sg, ids, 5) == 0
    host = ck.state_download(sg)
    for off, val in ((0, ord("X")), (80, 99), (12, 8)):
        bad = host.copy()
        bad[off] = val
        ck.state_upload(sg, bad)
        assert P.gpu.turn(sg, 1)[0] == 3
    other = pairs["gqa"]
    ck.state_upload(sg, host)
    assert other.gpu.turn(sg, 1)[0] == 3                            # another model's state


def test_cross_target_resume(ck, pairs):
    """A run continues on either target from the other's state ("The resumable state")."""
    wl = MODELS["gqa"]
    P = pairs["gqa"]
    ids = synth.prompt_ids(wl.spec, wl.n_prompt)
    ref, _ = P.init(ck, ids, wl.steps)
    P.orc.turn(ref, 10_000)
    # GPU first, oracle finishes
    so, sg = P.init(ck, ids, wl.steps)
    P.gpu.turn(sg, 20)
    host = ck.state_download(sg)
    P.orc.turn(host, 10_000)
    compare_states(P.orc, ref, host, wl.n_prompt, wl.steps, "gpu then oracle", turns=False)
    # oracle first, GPU finishes
    P.orc.turn(so, 25)
    ck.state_upload(sg, so)
    rc, res = P.gpu.turn(sg, 10_000)
    assert rc == 0 and res["complete"]
    compare_states(P.orc, ref, ck.state_download(sg), wl.n_prompt, wl.steps, "oracle then gpu",
                   turns=False)


def test_argmax_kernel_first_of_ties(ck, pairs):
    P = pairs["tiny_ws"]
    spec = P.spec
    ids = synth.prompt_ids(spec, 3)
    sg = P.gpu.new_state(3, 4)
    assert P.gpu.init_state(sg, ids, 4) == 0
    host = ck.state_download(sg)
    lay = P.orc.layout(3, 4)
    rng = np.random.default_rng(3)
    for case in range(6):
        logits = rng.integers(-5, 5, spec.vocab).astype(np.int64)
        if case == 0:
            logits[:] = -7                                   # all equal: index 0
        elif case == 1:
            logits[[17, 300, 511]] = 2**62                   # ties at the top
        elif case == 2:
            logits[-1] = 2**63 - 1
        host[lay["logits"]:lay["logits"] + 8 * spec.vocab] = logits.view(np.uint8)
        ck.state_upload(sg, host)
        rc, idx = P.gpu.argmax(sg)
        assert rc == 0 and idx == oracle.argmax(logits) == int(np.argmax(logits))
        rc, lg = P.gpu.logits(sg)
        assert rc == 0 and np.array_equal(lg, logits)


def test_model_artifact_errors(ck):
    art = synth.build_artifact(synth.TINY_WS)
    bad = art.copy()
    bad[0] = ord("X")
    assert ck.Model.load(bad)[0] == 2
    assert ck.Model.load(art[:-64].copy())[0] == 2
    bad = art.copy()
    bad[8:12] = 0
    assert ck.Model.load(bad)[0] == 1


# ---------------------------------------------------------------- full-size sampled positions

def _resume_one(ck, spec, n_prompt, max_tokens, gpu_positions, check_positions, path="step"):
    """GPU runs `gpu_positions`, then the oracle and the GPU each run `check_positions` more
    from that same state; every buffer of the two results must be identical."""
    P = Pair(ck, spec, path)
    ids = synth.prompt_ids(spec, n_prompt)
    sg = P.gpu.new_state(n_prompt, max_tokens)
    assert P.gpu.init_state(sg, ids, max_tokens) == 0
    if gpu_positions:
        rc, _ = P.gpu.turn(sg, gpu_positions)
        assert rc == 0
    host = ck.state_download(sg)
    rco, reso = P.orc.turn(host, check_positions)
    rcg, resg = P.gpu.turn(sg, check_positions)
    assert rco == rcg == 0 and reso["work"] == resg["work"] == check_positions
    got = ck.state_download(sg)
    compare_states(P.orc, host, got, n_prompt, max_tokens, f"{spec.name} sampled", turns=False)
    return oracle.header(got)


@pytest.mark.parametrize("path", list(PATHS))
def test_llama7b_shape_sampled_positions(ck, path):
    """7B-shaped model at full size, in the launch configuration bench.py times: two prompt
    positions on the GPU, then the first generating position (classifier and maximum pass
    included) on both targets."""
    h = _resume_one(ck, synth.LLAMA7B, n_prompt=3, max_tokens=4, gpu_positions=2, check_positions=1,
                    path=path)
    assert h["generated"] == 1


@pytest.mark.parametrize("path", list(PATHS))
def test_llama7b_bench_positions(ck, path):
    """The benchmark's own run at full size: the 7B-shaped model, its 128 prompt ids run on
    the GPU as bench.py runs them (127 layer-major, then the position that generates the
    first token), the state sized for the workload's 256 tokens; then generating positions
    128 and 129 on both targets from the GPU's state, every buffer and the working vectors
    the path writes compared after each."""
    spec = synth.LLAMA7B
    n_prompt, max_tokens = 128, 256
    P = Pair(ck, spec, path)
    ids = synth.prompt_ids(spec, n_prompt, run=0)
    sg = P.gpu.new_state(n_prompt, max_tokens)
    assert P.gpu.init_state(sg, ids, max_tokens) == 0
    rc, res = P.gpu.turn(sg, n_prompt - 1)
    assert rc == 0 and res["work"] == n_prompt - 1
    rc, res = P.gpu.turn(sg, 1)
    assert rc == 0 and res["generated"] == 1
    host = ck.state_download(sg)
    for pos in (n_prompt, n_prompt + 1):
        rco, reso = P.orc.turn(host, 1)
        rcg, resg = P.gpu.turn(sg, 1)
        assert rco == rcg == 0 and reso == resg, (pos, reso, resg)
        compare_states(P.orc, host, ck.state_download(sg), n_prompt, max_tokens, f"7B position {pos}",
                       vectors=VECTORS[path])
    assert oracle.header(host)["generated"] == 3


@pytest.mark.parametrize("path", list(PATHS))
def test_1b_long_context_sampled_position(ck, path):
    """1B-shaped model at 8192 context: 7936 prompt ids prefilled on the GPU position by
    position, then one generating position with attention over 7936 cached positions
    checked against the oracle."""
    wl = synth.WORKLOADS["1b_long"]
    h = _resume_one(ck, wl.spec, n_prompt=wl.n_prompt, max_tokens=wl.steps,
                    gpu_positions=wl.n_prompt - 1, check_positions=1, path=path)
    assert h["generated"] == 1 and h["position"] == wl.n_prompt


# (dim, heads, kv_heads): head sizes 128, 32 (grouped), 16, 8 and 4
LONG_ATTENTION = [(256, 2, 2), (256, 8, 4), (64, 4, 4), (64, 8, 8), (64, 16, 16)]


@pytest.mark.parametrize("dim,heads,kv_heads", LONG_ATTENTION)
def test_long_cache_attention_kernel(ck, dim, heads, kv_heads):
    """The per-phase attention kernel over 1060 cached positions (each cluster CTA walks about
    133 of them, several unrolled load batches): 1059 prompt positions on the GPU, then the
    generating position against the oracle, every buffer, at head sizes 128 to 4."""
    spec = synth.ModelSpec(f"long_attention_{dim}_{heads}_{kv_heads}", dim, 172, 2, heads, kv_heads, 512,
                           1100, scale_rule="well", tied=False, seed=0x5EED0031)
    h = _resume_one(ck, spec, n_prompt=1060, max_tokens=8, gpu_positions=1059, check_positions=1,
                    path="kernels")
    assert h["generated"] == 1


def test_1b_sixty_four_runs_sampled(ck):
    """The 1B-shaped model with 64 independent runs (64 prompt ids each, own state and
    cache), advanced in turns interleaved like a serving loop; sampled runs then take one
    generating position on both targets from the same state."""
    wl = synth.WORKLOADS["1b_x64"]
    spec = wl.spec
    art = synth.build_artifact(spec)
    orc = oracle.Model(art)
    rc, gpu = ck.Model.load(art)
    assert rc == 0
    states = []
    for r in range(wl.runs):
        ids = synth.prompt_ids(spec, wl.n_prompt, run=r)
        sg = gpu.new_state(wl.n_prompt, wl.steps)
        assert gpu.init_state(sg, ids, wl.steps) == 0
        states.append(sg)
    chunk = 16
    for done in range(0, wl.n_prompt - 1, chunk):  # the prompts, 16 positions a turn per run
        for sg in states:
            rc, res = gpu.turn(sg, min(chunk, wl.n_prompt - 1 - done))
            assert rc == 0, rc
    for r in (0, 37, wl.runs - 1):
        host = ck.state_download(states[r])
        rco, reso = orc.turn(host, 1)
        rcg, resg = gpu.turn(states[r], 1)
        assert rco == rcg == 0 and reso == resg, (r, reso, resg)
        compare_states(orc, host, ck.state_download(states[r]), wl.n_prompt, wl.steps, f"run {r}", turns=False)
        assert oracle.header(host)["generated"] == 1


# ---------------------------------------------------------------- layer-major prefill

MEDIUM = synth.ModelSpec("medium_gqa", 640, 1728, 2, 10, 5, 1000, 600, scale_rule="well", tied=False,
                         seed=0x5EED0041)


@pytest.mark.parametrize("chunk", [256, 7, 2])
def test_prefill_matches_the_oracle(ck, chunk):
    """Layer-major prefill of 299 prompt positions in chunks (the last one ragged) on a model
    whose matrices span several row tiles, more than four column groups (the f32 sums move
    to integers mid-row) and a padded last group; then the generating positions.  The whole
    state against the oracle run position by position."""
    P = Pair(ck, MEDIUM, "step")
    assert P.gpu.set_prefill(chunk) == 0
    n_prompt, steps = 300, 4
    ids = synth.prompt_ids(MEDIUM, n_prompt)
    so, sg = P.init(ck, ids, steps)
    rco, reso = P.orc.turn(so, n_prompt - 1)
    rcg, resg = P.gpu.turn(sg, n_prompt - 1)
    assert rco == rcg == 0 and reso == resg, (reso, resg)
    compare_states(P.orc, so, ck.state_download(sg), n_prompt, steps, f"prefill chunk {chunk}")
    rco, reso = P.orc.turn(so, 100)
    rcg, resg = P.gpu.turn(sg, 100)
    assert rco == rcg == 0 and reso == resg
    compare_states(P.orc, so, ck.state_download(sg), n_prompt, steps, f"after prefill {chunk}")


@pytest.mark.parametrize("path", list(PATHS))
def test_prefill_small_models(ck, path):
    """Every small model prefilled in one turn, at the default chunk and at chunks of 3,
    then generated to the end, against the oracle."""
    for name, wl in MODELS.items():
        for chunk in (256, 3):
            P = Pair(ck, wl.spec, path)
            assert P.gpu.set_prefill(chunk) == 0
            ids = synth.prompt_ids(wl.spec, wl.n_prompt)
            so, sg = P.init(ck, ids, wl.steps, temperature_q16=3 << 15, seed=chunk)
            for n in (wl.n_prompt - 1, 1000):
                rco, reso = P.orc.turn(so, n)
                rcg, resg = P.gpu.turn(sg, n)
                assert rco == rcg == 0 and reso == resg, (name, chunk, reso, resg)
                compare_states(P.orc, so, ck.state_download(sg), wl.n_prompt, wl.steps,
                               f"{name} chunk {chunk} after {n}")


@pytest.mark.parametrize("chunk", [256, 3])
def test_prefill_failure_matches_the_oracle(ck, chunk):
    """The literal tiny workload overflows a key store at position 1 (layer 1): the
    layer-major prefill fails the state at the same position with the same key."""
    wl = synth.WORKLOADS["tiny"]
    P = Pair(ck, wl.spec, "step")
    assert P.gpu.set_prefill(chunk) == 0
    ids = synth.prompt_ids(wl.spec, wl.n_prompt)
    so, sg = P.init(ck, ids, wl.steps)
    rco, reso = P.orc.turn(so, 100)
    rcg, resg = P.gpu.turn(sg, 100)
    assert rco == rcg == 8 and reso == resg, (reso, resg)
    assert resg["err_position"] == 1
    ho, hg = oracle.header(so), oracle.header(ck.state_download(sg))
    for k in ("phase", "error", "err_key", "position", "generated"):
        assert ho[k] == hg[k], k
    assert P.gpu.turn(sg, 1)[0] == 3
    assert P.gpu.set_prefill(4097) == 10


def _prefill_sampled(ck, spec, n_prompt, samples, chunk=256):
    """The GPU prefills n_prompt - 1 positions layer-major; for each sampled position p the
    oracle recomputes p alone from the GPU's cache below p (the words of p cleared first),
    and the key and value words of p in every layer must be identical, as must the last
    prefilled position's residual."""
    P = Pair(ck, spec, "step")
    assert P.gpu.set_prefill(chunk) == 0
    ids = synth.prompt_ids(spec, n_prompt)
    sg = P.gpu.new_state(n_prompt, 2)
    assert P.gpu.init_state(sg, ids, 2) == 0
    rc, res = P.gpu.turn(sg, n_prompt - 1)
    assert rc == 0 and res["work"] == n_prompt - 1
    got = ck.state_download(sg)
    lay = P.orc.layout(n_prompt, 2)
    cache, hd = n_prompt + 1, spec.head_dim
    for p in samples:
        host = got.copy()
        host[oracle.H_POSITION:oracle.H_POSITION + 4] = np.array([p], "<u4").view(np.uint8)
        words = []
        for name in ("k", "v"):
            for l in range(spec.layers):
                for kvh in range(spec.kv_heads):  # head-major: [layer][kv head][position][element]
                    o = lay[name] + 4 * (((l * spec.kv_heads + kvh) * cache + p) * hd)
                    host[o:o + 4 * hd] = 0
                    words.append((name, l, o))
        rco, reso = P.orc.turn(host, 1)
        assert rco == 0 and reso["work"] == 1
        for name, l, o in words:
            a, b = host[o:o + 4 * hd], got[o:o + 4 * hd]
            assert np.array_equal(a, b), (spec.name, p, name, l, np.flatnonzero(a != b)[:8])
        if p == n_prompt - 2:
            d = spec.dim
            assert np.array_equal(host[lay["x"]:lay["x"] + 8 * d], got[lay["x"]:lay["x"] + 8 * d])


def test_prefill_1b_shape_sampled_positions(ck):
    """1B-shaped model at full size: 299 prompt positions layer-major (chunks of 256 and 43),
    sampled positions from both chunks recomputed by the oracle."""
    _prefill_sampled(ck, synth.ONE_B, 300, [0, 131, 255, 256, 298])


def test_prefill_llama7b_shape_sampled_positions(ck):
    """7B-shaped model at full size: 69 prompt positions in one ragged chunk, the first and
    last recomputed by the oracle."""
    _prefill_sampled(ck, synth.LLAMA7B, 70, [0, 68])


# ---------------------------------------------------------------- many runs in one pass

def test_batched_runs_match_the_oracle(ck):
    """Five runs of one model with different prompts, lengths, temperatures and seeds,
    advanced one position each per batched pass from their first position to the end (runs
    finish at different passes and then drop out); every run's state against the oracle
    after every pass."""
    wl = MODELS["gqa"]
    P = Pair(ck, wl.spec, "step")
    runs = []
    for r, (n_prompt, steps, temp, seed) in enumerate([(12, 40, 0, 0), (3, 20, 1 << 16, 9),
                                                         (30, 8, 16 << 16, 0), (1, 30, 3 << 14, 77),
                                                         (7, 45, 0, 0)]):
        ids = synth.prompt_ids(wl.spec, n_prompt, run=r)
        so, sg = P.init(ck, ids, steps, temperature_q16=temp, seed=seed)
        runs.append([so, sg, n_prompt, steps])
    passes = 0
    while True:
        live = [r for r in runs if oracle.header(r[0])["phase"] == oracle.PHASE_RUNNING]
        if not live:
            break
        rc, res, rcs = P.gpu.turn_batch([r[1] for r in live])
        assert rc == 0 and rcs == [0] * len(live), (rc, rcs)
        for r, got in zip(live, res):
            rco, reso = P.orc.turn(r[0], 1)
            assert rco == 0 and reso == got, (passes, reso, got)
            compare_states(P.orc, r[0], ck.state_download(r[1]), r[2], r[3], f"pass {passes}")
        passes += 1
    assert passes == 51
    # complete states are refused one by one, the others in the same call still run
    so, sg = P.init(ck, synth.prompt_ids(wl.spec, 4), 3)
    rc, res, rcs = P.gpu.turn_batch([runs[0][1], sg])
    assert rc == 3 and rcs == [3, 0] and res[1]["work"] == 1
    assert P.gpu.turn_batch([sg, sg])[0] == 10                      # the same state twice


def test_batched_pass_graphs_across_bounds_counts_and_scratch_changes(ck):
    """The batched pass replays a CUDA graph captured per row count and position bound (the
    largest position rounded up to a multiple of 128): runs whose positions cross 128,
    passes that alternate between all runs and two of them, and a change of the prefill
    chunk (which frees the scratch the graphs point into) between passes; every run's state
    against the oracle after every pass it takes part in."""
    wl = MODELS["gqa"]
    P = Pair(ck, wl.spec, "kernels")
    runs = []
    for r, (n_prompt, steps) in enumerate([(120, 24), (100, 40), (126, 12)]):
        ids = synth.prompt_ids(wl.spec, n_prompt, run=r)
        so, sg = P.init(ck, ids, steps)
        rco, _ = P.orc.turn(so, n_prompt - 1)
        rcg, _ = P.gpu.turn(sg, n_prompt - 1)
        assert rco == rcg == 0
        runs.append([so, sg, n_prompt, steps])
    positions = set()
    for i in range(30):
        live = [r for r in runs if oracle.header(r[0])["phase"] == oracle.PHASE_RUNNING]
        if not live:
            break
        if i % 3 == 1:
            live = live[:2]
        if i == 12:
            assert P.gpu.set_prefill(64) == 0
        rc, res, rcs = P.gpu.turn_batch([r[1] for r in live])
        assert rc == 0 and rcs == [0] * len(live), (i, rc, rcs)
        for r, got in zip(live, res):
            positions.add(oracle.header(r[0])["position"])
            rco, reso = P.orc.turn(r[0], 1)
            assert rco == 0 and reso == got, (i, reso, got)
            compare_states(P.orc, r[0], ck.state_download(r[1]), r[2], r[3], f"pass {i}")
    assert min(positions) < 128 <= max(positions)


def test_batched_runs_fail_like_the_oracle(ck):
    """Literal tiny runs overflow their caches at different positions: each failing run
    fails alone, with the oracle's key, in the pass that reaches it, while the others go
    on."""
    wl = synth.WORKLOADS["tiny"]
    P = Pair(ck, wl.spec, "step")
    runs = []
    for r in range(4):
        ids = synth.prompt_ids(wl.spec, 2 + r, run=r)
        so, sg = P.init(ck, ids, 6)
        runs.append((so, sg))
    for _ in range(12):
        live = [r for r in runs if oracle.header(r[0])["phase"] == oracle.PHASE_RUNNING]
        if not live:
            break
        rc, res, rcs = P.gpu.turn_batch([r[1] for r in live])
        for (so, sg), got, rcg in zip(live, res, rcs):
            rco, reso = P.orc.turn(so, 1)
            assert rco == rcg and reso == got, (rco, rcg, reso, got)
            ho, hg = oracle.header(so), oracle.header(ck.state_download(sg))
            for k in ("phase", "error", "err_key", "position", "generated", "turns"):
                assert ho[k] == hg[k], k
    # this seed: three runs fail (positions 1, 0 and 6) and one completes
    assert [oracle.header(r[0])["phase"] for r in runs] == [oracle.PHASE_FAILED] * 3 + [oracle.PHASE_DONE]


def test_1b_sixty_four_runs_batched_sampled(ck):
    """The 1B-shaped model with 64 runs: prompts prefilled per run, then generating
    positions of all 64 runs in batched passes; sampled runs recomputed by the oracle for
    the last pass from the state before it."""
    wl = synth.WORKLOADS["1b_x64"]
    spec = wl.spec
    art = synth.build_artifact(spec)
    orc = oracle.Model(art)
    rc, gpu = ck.Model.load(art)
    assert rc == 0
    states = []
    for r in range(wl.runs):
        ids = synth.prompt_ids(spec, wl.n_prompt, run=r)
        sg = gpu.new_state(wl.n_prompt, wl.steps)
        assert gpu.init_state(sg, ids, wl.steps, temperature_q16=(r % 3) << 15, seed=r) == 0
        assert gpu.turn(sg, wl.n_prompt - 1)[0] == 0
        states.append(sg)
    for _ in range(3):
        rc, res, rcs = gpu.turn_batch(states)
        assert rc == 0 and all(x["generated_this_turn"] == 1 for x in res)
    snaps = {r: ck.state_download(states[r]) for r in (0, 1, 2, 37, wl.runs - 1)}
    rc, res, rcs = gpu.turn_batch(states)
    assert rc == 0
    for r, host in snaps.items():
        rco, reso = orc.turn(host, 1)
        assert rco == 0 and reso == res[r], (r, reso, res[r])
        compare_states(orc, host, ck.state_download(states[r]), wl.n_prompt, wl.steps, f"run {r}", turns=False)


# ---------------------------------------------------------------- text in, text out

@pytest.mark.parametrize("temp", [0, 3 << 15])
def test_text_prompt_to_text_output(ck, temp):
    """A text prompt through the library's tokenizer (phases 0 to 2), the GPU run, and the
    text of the generated tokens, against the oracle's tokenizer, run and text."""
    wl = MODELS["gqa"]
    spec = wl.spec
    blob = synth.tokenizer_blob(spec.vocab, spec.seed)
    rc, tok = ck.Tokenizer.load(blob, spec.vocab)
    assert rc == 0
    v = oracle.Vocab(blob, spec.vocab)
    text = synth.prompt_text(20, spec.seed, 3, blob)
    rcg, ids = tok.encode(text)
    rco, ids_o = v.encode(text)
    assert rcg == rco == 0 and ids.tolist() == ids_o
    P = Pair(ck, spec, "step")
    steps = 24
    so, sg = P.init(ck, ids, steps, temperature_q16=temp, seed=5)
    rco, reso = P.orc.turn(so, 10_000)
    rcg, resg = P.gpu.turn(sg, 10_000)
    assert rco == rcg == 0 and reso == resg
    compare_states(P.orc, so, ck.state_download(sg), len(ids), steps, "text run")
    rc, out = P.gpu.output_tokens(sg)
    assert rc == 0 and len(out) == steps
    rc, got = tok.decode(out, prev=int(ids[-1]))
    assert rc == 0 and got == v.decode(list(out), prev=int(ids[-1]))


@pytest.mark.parametrize("stride", [7, 1])
def test_page_state_round_trip_with_mid_layer_stops(ck, stride):
    """A text prompt run on the GPU into its generating positions; the state converted into
    the page's CURTAST2 state; the oracle's page executor runs it on in stops of `stride`
    steps (mid-layer and mid-attention) for two more positions; converted back at a position
    boundary, the GPU finishes the run.  Every byte equals the oracle's ids-mode run."""
    wl = MODELS["gqa"]
    spec = wl.spec
    blob = synth.tokenizer_blob(spec.vocab, spec.seed)
    rc, tok = ck.Tokenizer.load(blob, spec.vocab)
    assert rc == 0
    v = oracle.Vocab(blob, spec.vocab)
    text = synth.prompt_text(10, spec.seed, 2, blob)
    rc, ids = tok.encode(text)
    assert rc == 0
    steps = 12
    P = Pair(ck, spec, "step")
    so, sg = P.init(ck, ids, steps, flags=ck.CK_FLAG_STOP_TOKENS, temperature_q16=3 << 15, seed=21)
    rco, _ = P.orc.turn(so, 10**6)
    assert rco == 0
    rc, _ = P.gpu.turn(sg, len(ids))                  # the prompt and the first token
    assert rc == 0
    rc, page = P.gpu.state_to_page(tok, ck.state_download(sg), text)
    assert rc == 0
    h0 = oracle.page_header(page)
    assert h0["phase"] == 3 and h0["position"] == len(ids)
    stops = 0
    while True:
        h = oracle.page_header(page)
        if h["phase"] == 20 or (h["phase"] == 3 and h["position"] >= h0["position"] + 2):
            break
        near = h["phase"] >= 17 and h["position"] == h0["position"] + 1
        rc, ran = oracle.page_turn(P.orc, v, page, 1 if near else stride)
        assert rc == 0 and ran >= 1
        stops += 1
        if stops % 5 == 2:
            assert h["phase"] in range(3, 20)            # really mid-position
    assert stops > 10
    rc, back = P.gpu.state_from_page(page, len(ids), steps)
    assert rc == 0
    ck.state_upload(sg, back)
    rc, _ = P.gpu.turn(sg, 10**6)
    assert rc == 0
    compare_states(P.orc, so, ck.state_download(sg), len(ids), steps, "page round trip", turns=False)
    # the page's output text is the decoded output
    hp = oracle.page_header(page)
    pl = oracle.page_layout(P.orc, len(text), steps)
    out = page[pl["out"]:pl["out"] + 4 * hp["generated"]].view("<u4").tolist()
    assert page[pl["text"]:pl["text"] + hp["text_bytes"]].tobytes() == tok.decode(out, prev=int(ids[-1]))[1]
    # not a position boundary: refused
    rc, page2 = P.gpu.state_to_page(tok, ck.state_download(sg), text)
    oracle.page_turn(P.orc, v, page2, 0)
    assert P.gpu.state_from_page(page2, len(ids), steps)[0] == 0          # done: a boundary
    rc, sg2 = P.init(ck, ids, steps, flags=ck.CK_FLAG_STOP_TOKENS)
    rc, page3 = P.gpu.state_to_page(tok, ck.state_download(sg2), text)
    assert rc == 0
    oracle.page_turn(P.orc, v, page3, 2)                # into position 0's layer 0
    assert P.gpu.state_from_page(page3, len(ids), steps)[0] == 3
    so4, sg4 = P.init(ck, ids, steps)                   # without the stop-token flag
    assert P.gpu.state_to_page(tok, ck.state_download(sg4), text)[0] == 3


def test_paths_agree_and_unknown_path_is_rejected(ck):
    wl = MODELS["gqa"]
    P = Pair(ck, wl.spec, "step")
    assert P.gpu.set_path(7) == 10
    ids = synth.prompt_ids(wl.spec, wl.n_prompt)
    outs = []
    for path in PATHS.values():
        assert P.gpu.set_path(path) == 0
        sg = P.gpu.new_state(wl.n_prompt, wl.steps)
        assert P.gpu.init_state(sg, ids, wl.steps) == 0
        rc, res = P.gpu.turn(sg, 10_000)
        assert rc == 0 and res["complete"]
        outs.append(ck.state_download(sg))
    lay = P.orc.layout(wl.n_prompt, wl.steps)
    for name, end in (("out", lay["x"]), ("x", lay["xb"]), ("logits", lay["scores"]), ("k", lay["size"])):
        assert np.array_equal(outs[0][lay[name]:end], outs[1][lay[name]:end]), name
