"""Lazy (early-exit) stochastic verification: the rows after the first
rejection are never read ("Speculative decoding: guess a few tokens first",
section "What happens in one round", step 3), yet tokens and accept counts
must equal the full pass bit for bit, and the oracle's within its margin.
Log-probabilities of the positions read are the full pass's exactly; later
positions are NaN."""
import numpy as np
import pytest

import oracle
from speculative_decoding_verification_59_gb300 import workloads as W

from parity import compare_sample

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def sv():
    import __graft_entry__
    __graft_entry__.build()
    import speculative_decoding_verification_59_gb300 as m
    return m


def dev_logits(a, dtype):
    t = torch.from_numpy(np.ascontiguousarray(a)).cuda()
    return t.to(torch.bfloat16) if dtype == "bf16" else t


def both(sv, x, u=None, ws=None):
    zt, zd = dev_logits(x.target, x.dtype), dev_logits(x.draft, x.dtype)
    xt = torch.from_numpy(x.draft_tokens).cuda()
    uu = torch.from_numpy(x.uniforms if u is None else u).cuda()
    full = sv.verify_sample(zt, zd, xt, uu, x.T, logprobs=True, workspace=ws)
    lazy = sv.verify_sample(zt, zd, xt, uu, x.T, logprobs=True, workspace=ws, lazy=True)
    torch.cuda.synchronize()
    return [t.cpu().numpy() for t in full], [t.cpu().numpy() for t in lazy]


def check_same(full, lazy):
    (tf, af, lf), (tl, al, ll) = full, lazy
    assert np.array_equal(tf, tl)
    assert np.array_equal(af, al)
    B, g = lf.shape[:2]
    for b in range(B):
        k = int(al[b])
        for i in range(g):
            if k >= 0 and i <= k:
                assert np.array_equal(lf[b, i], ll[b, i]), (b, i, lf[b, i], ll[b, i])
            else:
                assert np.isnan(ll[b, i]).all(), (b, i, ll[b, i])


@pytest.mark.parametrize("name,B,gamma,V", [
    ("chain-small", 1, 4, 1000),
    ("chain-small", 5, 0, 512),        # gamma = 0: only the bonus row
    ("chain-b8", 8, 7, 151936),
    ("chain-b64", 64, 7, 151936),
    ("chain-b256", 256, 4, 128256),
    ("chain-b8", 3, 5, 20011),         # rows not a multiple of 16 bytes: full pass, same outputs
    ("chain-b256", 4, 3, 7001),
])
def test_lazy_equals_full_and_oracle(sv, name, B, gamma, V):
    x = W.make_chain(name, B=B, gamma=gamma, V=V)
    rng = np.random.default_rng(B * 7 + V)
    for rnd in range(3):
        u = x.uniforms if rnd == 0 else rng.random((x.B, x.gamma + 1), dtype=np.float32)
        full, lazy = both(sv, x, u)
        check_same(full, lazy)
        ref = oracle.verify_sample(x.target, x.draft, x.draft_tokens, u, x.T, want_ratio=True,
                                   want_cdf=True)
        res = compare_sample(lazy[0], lazy[1], ref, x.draft_tokens, u)
        assert not res["failures"], res["failures"][:5]


def test_lazy_bad_tokens_and_reuse(sv):
    x = W.make_chain("chain-b8", B=4, gamma=3, V=8192)
    x.draft_tokens = x.draft_tokens.copy()
    x.draft_tokens[2, 1] = 8192                       # out of range: the sequence is bad
    ws = sv.Workspace()
    full, lazy = both(sv, x, ws=ws)
    check_same(full, lazy)
    assert lazy[1][2] == -1 and (lazy[0][2] == -1).all()
    assert ws.read_error() & sv.SPEC_DEVERR_TOKEN_RANGE
    x.draft_tokens[2, 1] = 5
    full, lazy = both(sv, x, ws=ws)                    # the same workspace, clean again
    check_same(full, lazy)
    assert ws.read_error() == 0


def test_lazy_identical_models_read_every_position(sv):
    x = W.make_chain("chain-b8", B=4, V=8192)
    x.draft = x.target[:, :x.gamma].copy()             # p = q: every draft accepted
    full, lazy = both(sv, x)
    check_same(full, lazy)
    assert (lazy[1] == x.gamma).all()


@pytest.fixture
def every_group(sv):
    """Split at every group boundary whatever the sizes (the library otherwise
    merges the groups of small problems into one pass); the built-in figure
    is restored afterwards."""
    sv.spec_verify_set_lazy_split_bytes(0)
    yield
    sv.spec_verify_set_lazy_split_bytes(-1.0)


@pytest.mark.parametrize("gamma", [1, 2, 5, 6, 13, 14, 30])
def test_lazy_group_boundaries(sv, every_group, gamma):
    """Positions go in groups [0, 2), [2, 6), [6, 14), [14, 30), ...: draft
    counts on either side of a boundary, with the chain-b64 generator's three
    draft-noise levels (acceptance from ~0.3 to ~0.9) and fresh uniforms."""
    x = W.make_chain("chain-b64", B=12, gamma=gamma, V=4096)
    rng = np.random.default_rng(gamma)
    for rnd in range(3):
        u = x.uniforms if rnd == 0 else rng.random((x.B, x.gamma + 1), dtype=np.float32)
        full, lazy = both(sv, x, u)
        check_same(full, lazy)
        ref = oracle.verify_sample(x.target, x.draft, x.draft_tokens, u, x.T, want_ratio=True,
                                   want_cdf=True)
        res = compare_sample(lazy[0], lazy[1], ref, x.draft_tokens, u)
        assert not res["failures"], res["failures"][:5]


def test_lazy_largest_gamma_every_group(sv, every_group):
    """gamma = 256 (the most drafts a call takes) with p = q: every draft is
    accepted, so all eight position groups run, the largest of 128 positions."""
    x = W.make_chain("chain-b8", B=2, gamma=256, V=2048)
    x.draft = x.target[:, :x.gamma].copy()
    full, lazy = both(sv, x)
    check_same(full, lazy)
    assert (lazy[1] == x.gamma).all()


def test_lazy_every_sequence_rejects_first_draft(sv, every_group):
    """The first draft is the target's least likely token, on which the draft
    model puts nearly all its mass (logit 40): p/q is ~0, so every sequence
    rejects it and the later groups run with empty survivor lists."""
    x = W.make_chain("chain-b8", B=6, gamma=7, V=8192)
    x.draft, x.draft_tokens = x.draft.copy(), x.draft_tokens.copy()
    for b in range(x.B):
        j = int(np.argmin(x.target[b, 0]))
        x.draft_tokens[b, 0] = j
        x.draft[b, 0, j] = 40.0
    full, lazy = both(sv, x)
    check_same(full, lazy)
    assert (lazy[1] == 0).all()


def test_lazy_empty_row_in_a_later_group(sv, every_group):
    """An all -inf target row at position 4 (the second group) of a sequence
    whose drafts before it are all accepted: the sequence is bad (-1), as in
    the full pass, and the error word says why."""
    x = W.make_chain("chain-b8", B=3, gamma=7, V=4096)
    x.draft = x.target[:, :x.gamma].copy()             # every draft accepted ...
    x.target = x.target.copy()
    x.target[1, 4, :] = -np.inf                        # ... until row 4 of sequence 1
    x.draft[1, 4, :] = -np.inf
    ws = sv.Workspace()
    full, lazy = both(sv, x, ws=ws)
    check_same(full, lazy)
    assert lazy[1][1] == -1 and (lazy[0][1] == -1).all()
    assert (lazy[1][[0, 2]] == x.gamma).all()
    assert ws.read_error() & sv.SPEC_DEVERR_EMPTY_ROW


@pytest.mark.parametrize("split", [0, 1e11])
def test_lazy_schedule_does_not_change_results(sv, split):
    """chain-b64 at full size with every boundary taken (three groups) and with
    none (one group): the same tokens, counts and log-probabilities as the
    full pass either way."""
    sv.spec_verify_set_lazy_split_bytes(split)
    try:
        x = W.make_chain("chain-b64")
        full, lazy = both(sv, x)
        check_same(full, lazy)
    finally:
        sv.spec_verify_set_lazy_split_bytes(-1.0)
