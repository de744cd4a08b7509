"""GPU parity: the CUDA path (through the C ABI) against the fp64 oracle on
the same seeded inputs.  Greedy and tree results are bit-exact; sampling is
exact except for differences the oracle's own margin (< 1e-4) excuses, and
those must stay under 0.01 % of rows."""
import numpy as np
import pytest

import oracle
from speculative_decoding_verification_59_gb300 import workloads as W

from parity import compare_exact, compare_sample

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

RATE_BAR = 1e-4


@pytest.fixture(scope="module")
def sv():
    import __graft_entry__
    __graft_entry__.build()
    import speculative_decoding_verification_59_gb300 as m
    return m


def dev_logits(a, dtype):
    t = torch.from_numpy(np.ascontiguousarray(a)).cuda()
    return t.to(torch.bfloat16) if dtype == "bf16" else t


def dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def run_sample(sv, x, logprobs=True, ws=None):
    tok, acc, lp = sv.verify_sample(dev_logits(x.target, x.dtype), dev_logits(x.draft, x.dtype),
                                    dev(x.draft_tokens), dev(x.uniforms), x.T, logprobs=True,
                                    workspace=ws)
    torch.cuda.synchronize()
    return tok.cpu().numpy(), acc.cpu().numpy(), lp.cpu().numpy()


def check_sample(sv, x, ws=None):
    tok, acc, lp = run_sample(sv, x, ws=ws)
    ref = oracle.verify_sample(x.target, x.draft, x.draft_tokens, x.uniforms, x.T,
                               want_logprob=True, want_ratio=True, want_cdf=True)
    res = compare_sample(tok, acc, ref, x.draft_tokens, x.uniforms, gpu_lp=lp)
    assert not res["failures"], res["failures"][:5]
    return res


def check_greedy(sv, target, dtype, tokens, ws=None):
    tok, acc = sv.verify_greedy(dev_logits(target, dtype), dev(tokens), workspace=ws)
    torch.cuda.synchronize()
    ref = oracle.verify_greedy(target, tokens)
    f = compare_exact("tokens", tok.cpu().numpy(), ref["tokens"]) + \
        compare_exact("accepted", acc.cpu().numpy(), ref["accepted"])
    assert not f, f
    return ref


def check_tree(sv, t, ws=None):
    nodes, tok, acc = sv.verify_tree_greedy(dev_logits(t.target, t.dtype), dev(t.node_tokens),
                                            dev(t.parents), workspace=ws)
    torch.cuda.synchronize()
    ref = oracle.verify_tree_greedy(t.target, t.node_tokens, t.parents)
    f = compare_exact("nodes", nodes.cpu().numpy(), ref["nodes"]) + \
        compare_exact("tokens", tok.cpu().numpy(), ref["tokens"]) + \
        compare_exact("accepted", acc.cpu().numpy(), ref["accepted"])
    assert not f, f
    return ref


# ------------------------------------------------------------------ greedy
@pytest.mark.parametrize("name,B,gamma,V", [
    ("chain-b8", 3, 4, 20011),       # bf16, V odd: unaligned rows, scalar path, ragged tail
    ("chain-b8", 2, 7, 40000),       # bf16, aligned, 3 block chunks with a ragged last one
    ("chain-b256", 5, 3, 7001),      # fp32, unaligned
    ("chain-b256", 4, 4, 9000),      # fp32, aligned, ragged
    ("chain-small", 1, 4, 1000),
    ("chain-small", 3, 0, 257),      # gamma = 0: bonus argmax only
    ("chain-small", 2, 3, 1),        # V = 1
])
def test_greedy_small(sv, name, B, gamma, V):
    x = W.make_chain(name, B=B, gamma=gamma, V=V)
    check_greedy(sv, x.target, x.dtype, x.greedy_tokens)
    check_greedy(sv, x.target, x.dtype, x.draft_tokens)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_greedy_ties_and_signed_zero(sv, dtype):
    rng = np.random.default_rng(0)
    B, gamma, V = 16, 5, 3000
    z = rng.integers(-2, 3, (B, gamma + 1, V)).astype(np.float32)      # massive ties
    z[0, 0, :] = -0.0
    z[0, 0, 5] = 0.0
    z[1, :, :] = -np.inf                                                # all -inf: index 0
    x = np.argmax(z[:, :gamma], axis=2).astype(np.int32)
    x[::3, 2] = (x[::3, 2] + 1) % V
    check_greedy(sv, z, dtype, x)


# -------------------------------------------------------------------- tree
@pytest.mark.parametrize("B,V,depth,branches", [(4, 5003, 7, 4), (3, 16384, 3, 2), (2, 999, 1, 0)])
def test_tree_small(sv, B, V, depth, branches):
    check_tree(sv, W.make_tree(B=B, V=V, depth=depth, branches=branches))


@pytest.mark.parametrize("N", [40, 200])
def test_tree_random_topologies_with_ties(sv, N):
    """Random parents, integer logits (massive argmax ties) and 80% of tokens
    equal to the parent's argmax, so sibling paths of equal length are common:
    the lowest node ids must win.  40 nodes take the decide kernel's sweep,
    200 its pointer-doubling walk."""
    rng = np.random.default_rng(N)
    B, V = 24, 600
    z = rng.integers(-2, 3, (B, N, V)).astype(np.float32)
    par = np.empty((B, N), np.int32)
    tok = np.empty((B, N), np.int32)
    for b in range(B):
        par[b, 0], tok[b, 0] = -1, -1
        g = np.argmax(z[b], axis=1)
        for n in range(1, N):
            par[b, n] = rng.integers(0, n)
            tok[b, n] = g[par[b, n]] if rng.random() < 0.8 else rng.integers(0, V)
    t = W.TreeInputs(z, tok, par, "f32", B, N, V, "random")
    check_tree(sv, t)
    t.dtype = "bf16"
    check_tree(sv, t)


# ------------------------------------------------------------------ sample
@pytest.mark.parametrize("name,B,gamma,V", [
    ("chain-b8", 4, 7, 20011),       # bf16 unaligned
    ("chain-b8", 3, 5, 48000),       # bf16 aligned, several tiles + ragged
    ("chain-b64", 6, 7, 30000),      # T = 0.6, three draft-noise levels
    ("chain-b256", 6, 4, 9001),      # fp32 unaligned
    ("chain-b256", 5, 4, 12000),     # fp32 aligned
    ("chain-small", 1, 4, 1000),
    ("chain-small", 4, 0, 500),      # gamma = 0: plain sampling from p_0
    ("chain-small", 3, 2, 1),        # V = 1
])
def test_sample_small(sv, name, B, gamma, V):
    check_sample(sv, W.make_chain(name, B=B, gamma=gamma, V=V))


@pytest.mark.parametrize("name,T", [
    ("chain-b8", 1e-3),     # sharp: most rows put almost all mass on one token
    ("chain-b8", 1e-12),    # extreme: the row-floor fast path is off, guarded exponentials
    ("chain-b8", 40.0),     # flat
    ("chain-b256", 1e-12),
])
def test_sample_extreme_temperatures(sv, name, T):
    check_sample(sv, W.make_chain(name, B=4, gamma=3, V=9000, T=T))


def test_sample_huge_logits(sv):
    # |max logit| >= 1e30 also switches the final pass to the guarded exponentials
    x = W.make_chain("chain-b256", B=4, gamma=3, V=9000)
    x.target = (x.target * np.float32(4e30)).astype(np.float32)
    x.draft = (x.draft * np.float32(4e30)).astype(np.float32)
    x.T = 3e30
    check_sample(sv, x)


def test_sample_identical_models_accept_all(sv):
    x = W.make_chain("chain-b8", B=4, V=8192)
    x.draft = x.target[:, :x.gamma].copy()
    tok, acc, _ = run_sample(sv, x)
    assert (acc == x.gamma).all()
    check_sample(sv, x)


def test_sample_bad_inputs_flagged(sv):
    x = W.make_chain("chain-b256", B=5, gamma=3, V=4096)
    x.draft_tokens = x.draft_tokens.copy()
    x.draft_tokens[1, 2] = 4096
    x.draft_tokens[2, 0] = -5
    x.target = x.target.copy()
    x.target[3, 1, :] = -np.inf
    ws = sv.Workspace()
    tok, acc, _ = run_sample(sv, x, ws=ws)
    assert list(acc[1:4]) == [-1, -1, -1] and (tok[1:4] == -1).all()
    code = ws.read_error()
    assert code & sv.SPEC_DEVERR_TOKEN_RANGE and code & sv.SPEC_DEVERR_EMPTY_ROW
    assert ws.read_error() == 0                              # cleared by the read
    check_sample(sv, x, ws=ws)
    ws.read_error()


@pytest.mark.parametrize("dtype,V", [("f32", 2), ("bf16", 16)])
def test_sample_residual_without_mass(sv, dtype, V):
    """Target [0, -58], draft [0, -46] on the first two tokens (the rest
    masked): the drafted token 1 is rejected and the residual's exact mass
    lies wholly on token 0, below what the working precision resolves.  Token
    0 must come out, no error is flagged, and the oracle agrees."""
    zt = np.full((1, 2, V), -np.inf, np.float32)
    zd = np.full((1, 1, V), -np.inf, np.float32)
    zt[0, 0, :2] = [0.0, -58.0]
    zt[0, 1, :2] = [0.0, -3.0]
    zd[0, 0, :2] = [0.0, -46.0]
    x = W.make_chain("chain-small", B=1, gamma=1, V=V)
    x.target, x.draft, x.dtype, x.T = zt, zd, dtype, 1.0
    x.draft_tokens = np.array([[1]], np.int32)
    ws = sv.Workspace()
    for u_final in (0.0, 0.3, 0.999999):
        x.uniforms = np.array([[0.5, u_final]], np.float32)
        tok, acc, _ = run_sample(sv, x, ws=ws)
        assert acc.tolist() == [0] and tok.tolist() == [[0, -1]]
        check_sample(sv, x, ws=ws)
    assert ws.read_error() == 0


def test_masked_tokens(sv):
    """-inf logits are masked tokens: never chosen, and q(x) = 0 accepts."""
    x = W.make_chain("chain-b256", B=6, gamma=3, V=2048)
    x.target = x.target.copy()
    x.draft = x.draft.copy()
    x.target[:, :, :1000] = -np.inf
    x.draft[:, :, 1000:1500] = -np.inf
    x.draft_tokens = np.full_like(x.draft_tokens, 1200)
    res = check_sample(sv, x)
    tok, acc, _ = run_sample(sv, x)
    assert (tok[tok >= 0] >= 1000).all()


def test_workspace_shared_across_modes_and_calls(sv):
    ws = sv.Workspace()
    a = W.make_chain("chain-b8", B=2, V=16384)
    t = W.make_tree(B=2, V=16384)
    for _ in range(2):
        check_sample(sv, a, ws=ws)
        check_greedy(sv, a.target, a.dtype, a.greedy_tokens, ws=ws)
        check_tree(sv, t, ws=ws)


def test_repeat_calls_are_bitwise_identical(sv):
    x = W.make_chain("chain-b64", B=8, V=65536)
    r1 = run_sample(sv, x)
    r2 = run_sample(sv, x)
    for a, b in zip(r1, r2):
        assert np.array_equal(a, b, equal_nan=True)


# ------------------------------------------------------ full-size workloads
@pytest.mark.parametrize("name", ["chain-small", "chain-b8", "chain-b64", "chain-b256"])
def test_full_size_sample(sv, name):
    """One call per workload at full size.  The rate itself is measured in
    test_gpu_rate.py over many draws; a single call may show at most ten times
    the count the rate bar allows on its rows, rounded down (0 for the three
    smaller workloads, 1 for the 1280 rows of chain-b256)."""
    x = W.make_chain(name)
    res = check_sample(sv, x)
    assert res["excused"] <= int(10 * RATE_BAR * res["rows"]), res["events"]


@pytest.mark.parametrize("name", ["chain-small", "chain-b8", "chain-b64", "chain-b256"])
def test_full_size_greedy(sv, name):
    x = W.make_chain(name)
    check_greedy(sv, x.target, x.dtype, x.draft_tokens)
    check_greedy(sv, x.target, x.dtype, x.greedy_tokens)


def test_full_size_tree(sv):
    check_tree(sv, W.make_tree("tree-b32"))


def test_split_stats_finish_equals_composite(sv):
    """spec_verify_sample == spec_verify_sample_stats then spec_verify_sample_finish."""
    x = W.make_chain("chain-b64", B=5, V=30000)
    zt, zd = dev_logits(x.target, x.dtype), dev_logits(x.draft, x.dtype)
    xt, u = dev(x.draft_tokens), dev(x.uniforms)
    tok1, acc1, lp1 = sv.verify_sample(zt, zd, xt, u, x.T, logprobs=True)
    ws = sv.Workspace()
    wp, wb = ws.get(x.B, x.gamma, x.V)
    tok2 = torch.full_like(tok1, -7)
    acc2 = torch.full_like(acc1, -7)
    lp2 = torch.zeros_like(lp1)
    st = torch.cuda.current_stream().cuda_stream
    code = sv.SPEC_DTYPE_BF16
    assert sv.spec_verify_sample_stats(zt.data_ptr(), zd.data_ptr(), code, x.T, x.B, x.gamma, x.V,
                                       wp, wb, st) == sv.SPEC_OK
    assert sv.spec_verify_sample_finish(zt.data_ptr(), zd.data_ptr(), code, xt.data_ptr(),
                                        u.data_ptr(), x.T, x.B, x.gamma, x.V, tok2.data_ptr(),
                                        acc2.data_ptr(), lp2.data_ptr(), wp, wb, st) == sv.SPEC_OK
    torch.cuda.synchronize()
    assert torch.equal(tok1, tok2) and torch.equal(acc1, acc2) and torch.equal(lp1, lp2)


def test_sample_largest_vocabulary_and_beyond(sv):
    """A vocabulary of 1M works; above 2097152 (256 chunks of 8192, the most
    the search kernel scans) the call is refused with SPEC_ERR_INVALID_ARG."""
    x = W.make_chain("chain-b8", B=1, gamma=2, V=1 << 20)
    check_sample(sv, x)
    big = 2097153
    fake = 1 << 20
    ws = sv.Workspace()
    wp, wb = ws.get(1, 1, big)
    st = sv.spec_verify_sample(fake, fake, sv.SPEC_DTYPE_BF16, fake, fake, 1.0, 1, 1, big, fake,
                               fake, None, wp, wb, None)
    assert st == sv.SPEC_ERR_INVALID_ARG


def test_sample_batch_beyond_grid_y_limit(sv):
    """More sequences than a grid's y dimension holds (65535): the final-pass
    kernel numbers its CTAs along x only."""
    x = W.make_chain("chain-b256", B=70000, gamma=1, V=24)
    res = check_sample(sv, x)
    assert res["rows"] == 70000 * 2


def test_no_device_error_on_valid_inputs(sv):
    """Valid calls of every mode leave the device error word clear (no bad
    input, and no bounded wait inside a kernel ever ran out)."""
    ws = sv.Workspace()
    a = W.make_chain("chain-b64", B=8, V=151936)
    t = W.make_tree(B=4, V=151936)
    check_sample(sv, a, ws=ws)
    check_greedy(sv, a.target, a.dtype, a.draft_tokens, ws=ws)
    check_tree(sv, t, ws=ws)
    assert ws.read_error() == 0


# ------------------------------------------------------- largest and empty sizes
def test_sample_largest_gamma(sv):
    # gamma = 256 is the most a sampling call takes (2 * 256 + 1 rows per sequence)
    x = W.make_chain("chain-b8", B=2, gamma=256, V=4096)
    res = check_sample(sv, x)
    assert res["rows"] == 2 * 257


def test_greedy_longest_chain(sv):
    # gamma + 1 = 1024 rows, drafts equal to the target argmax for long runs
    x = W.make_chain("chain-b8", B=2, gamma=1023, V=2048)
    am = np.argmax(x.target[:, :x.gamma], axis=2).astype(np.int32)
    tokens = am.copy()
    tokens[0, 700] = (tokens[0, 700] + 1) % x.V          # sequence 0 stops at 700, 1 accepts all
    ref = check_greedy(sv, x.target, x.dtype, tokens)
    assert ref["accepted"].tolist() == [700, 1023]


@pytest.mark.parametrize("depth,branches,match", [(31, 32, 0.9), (1023, 0, 1.0), (1023, 0, 0.995)])
def test_tree_largest(sv, depth, branches, match):
    """1024 nodes, the most a tree call takes: 1 + 31 + 31 * 32 (wide and shallow),
    or a chain of 1023 below the root, every node accepted (the walk is 1023
    long) or a few mismatches along it."""
    t = W.make_tree(B=2, V=2048, depth=depth, branches=branches, match_prob=match)
    assert t.node_tokens.shape[1] == 1024
    check_tree(sv, t)


def test_empty_batch(sv):
    x = W.make_chain("chain-small", B=1)
    zt = dev_logits(x.target[:0], x.dtype)
    zd = dev_logits(x.draft[:0], x.dtype)
    tok, acc = sv.verify_sample(zt, zd, dev(x.draft_tokens[:0]), dev(x.uniforms[:0]), x.T)
    assert tok.shape == (0, x.gamma + 1) and acc.shape == (0,)
    tok, acc = sv.verify_greedy(zt, dev(x.draft_tokens[:0]))
    assert tok.shape == (0, x.gamma + 1)


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_sample_many_equal_ratios(sv, dtype):
    """Integer logits: thousands of elements share each ratio p_j/q_j, the case
    where the residual sums' first-order move from the approximate to the exact
    normaliser ratio could miss the most mass."""
    rng = np.random.default_rng(17)
    B, g, V = 48, 3, 24576
    zt = rng.integers(-3, 4, size=(B, g + 1, V)).astype(np.float32)
    zd = zt[:, :g] + rng.integers(-1, 2, size=(B, g, V)).astype(np.float32)
    x = W.make_chain("chain-b256" if dtype == "f32" else "chain-b8", B=B, gamma=g, V=V)
    x.target, x.draft = zt, zd
    for r in range(4):
        x.uniforms = rng.random((B, g + 1), dtype=np.float32)
        check_sample(sv, x)


@pytest.mark.parametrize("name,V", [("chain-b8", 8), ("chain-b8", 16), ("chain-b8", 24),
                                    ("chain-b256", 4), ("chain-b256", 8)])
def test_rows_of_one_to_three_vectors(sv, name, V):
    """Rows of 16 to 48 bytes take the bulk-copy ring (their length is a
    multiple of 16): a stage and a warp chunk hold a few bytes, the rest of the
    warp chunk reads as -inf.  Sampling, lazy sampling, greedy and tree
    verification against the oracle."""
    x = W.make_chain(name, B=5, gamma=3, V=V)
    check_sample(sv, x)
    tok, acc = sv.verify_sample(dev_logits(x.target, x.dtype), dev_logits(x.draft, x.dtype),
                                dev(x.draft_tokens), dev(x.uniforms), x.T, lazy=True)
    full = run_sample(sv, x)
    torch.cuda.synchronize()
    assert np.array_equal(tok.cpu().numpy(), full[0]) and np.array_equal(acc.cpu().numpy(), full[1])
    check_greedy(sv, x.target, x.dtype, x.greedy_tokens)
    check_tree(sv, W.make_tree(B=3, V=V, depth=3, branches=2))
