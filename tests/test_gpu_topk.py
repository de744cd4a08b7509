"""GPU parity of the top-K branch tokens (AdaPLD section 3.3, Algorithm 1:
TopKNextTokens minus the main path's first token) against the oracle: token
lists and their logits must be bit-exact, including the order of equal
logits (lower index first) and the -1 padding."""
import numpy as np
import pytest

import oracle
from speculative_decoding_verification_59_gb300 import workloads as W

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def sv():
    import __graft_entry__
    __graft_entry__.build()
    import speculative_decoding_verification_59_gb300 as m
    return m


def run(sv, z, K, ex, dtype, ws=None):
    t = torch.from_numpy(np.ascontiguousarray(z)).cuda()
    if dtype == "bf16":
        t = t.to(torch.bfloat16)
    e = None if ex is None else torch.from_numpy(np.ascontiguousarray(ex, dtype=np.int32)).cuda()
    idx, val = sv.topk_exclude(t, K, e, values=True, workspace=ws)
    torch.cuda.synchronize()
    return idx.cpu().numpy(), val.cpu().numpy()


def check(sv, z, K, ex, dtype, ws=None):
    z = np.ascontiguousarray(z, dtype=np.float32)
    if dtype == "bf16":
        z = W.to_bf16_exact(z)            # both sides see the same bf16 values (+-inf stay)
    R, V = z.shape
    idx, val = run(sv, z, K, ex, dtype, ws)
    ref = oracle.topk_exclude(z, K, ex)
    bad = np.argwhere(idx != ref["idx"])
    assert bad.size == 0, (bad[:3], idx[bad[0][0]], ref["idx"][bad[0][0]])
    assert np.array_equal(val, ref["val"]), "values differ"
    return ref


def exclusions(rng, z, K):
    """-1, a token of the row's top K, or an out-of-range value, by row."""
    R, V = z.shape
    top = oracle.topk_exclude(z, K)["idx"]
    ex = np.full(R, -1, np.int32)
    for r in range(R):
        m = r % 4
        if m == 1:
            ex[r] = top[r, r % K] if top[r, r % K] >= 0 else -1
        elif m == 2:
            ex[r] = rng.integers(0, V)
        elif m == 3:
            ex[r] = V + 5 if r % 8 == 3 else -7
    return ex


def tied_rows(rng, R, V):
    # integer logits in a narrow range: many equal values, all exact in bf16
    return rng.integers(-6, 6, size=(R, V)).astype(np.float32)


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("V", [1, 5, 1000, 20011, 40000, 151936])
@pytest.mark.parametrize("K", [1, 3, 4, 8])
def test_topk_ties_and_exclusions(sv, dtype, V, K):
    rng = np.random.default_rng(V * 10 + K)
    R = 24 if V < 100000 else 9
    z = tied_rows(rng, R, V)
    check(sv, z, K, exclusions(rng, z, K), dtype)


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_topk_gaussian_rows_without_exclusion(sv, dtype):
    x = W.make_chain("chain-b8" if dtype == "bf16" else "chain-b256", B=6, gamma=3, V=30000)
    z = x.target.reshape(-1, x.V)
    for K in (2, 4, 5, 8):
        check(sv, z, K, None, dtype)


def test_topk_masked_and_signed_zero(sv):
    V = 4096
    z = np.zeros((6, V), np.float32)
    z[0, :] = -np.inf                                  # fully masked: index order
    z[1, :] = -np.inf
    z[1, [17, 900, 4000]] = [1.0, 3.0, 1.0]            # 3 finite logits, then masked ones
    z[2, ::2] = -0.0                                   # +0 and -0 everywhere: index order
    z[3, :] = -np.inf
    z[3, 5] = 0.0                                      # one finite logit, K = 4 of -inf after it
    z[4] = np.linspace(-1, 1, V, dtype=np.float32)
    z[4, 100] = np.inf                                 # +inf is an ordinary largest value
    z[5] = np.arange(V, dtype=np.float32)[::-1]        # strictly decreasing
    ex = np.array([0, 900, 2, -1, 100, 1], np.int32)
    for dtype in ("bf16", "f32"):
        check(sv, z, 4, ex, dtype)


def test_topk_full_size_tree_rows(sv):
    # every node row of the tree-b32 workload: 1152 rows of 151936 bf16 logits
    t = W.make_tree("tree-b32")
    z = t.target.reshape(-1, t.V)
    rng = np.random.default_rng(5)
    ex = exclusions(rng, z, 4)
    check(sv, z, 4, ex, "bf16")


def test_topk_workspace_reuse_and_repeat(sv):
    ws = sv.Workspace()
    rng = np.random.default_rng(9)
    z1 = tied_rows(rng, 50, 20000)
    z2 = tied_rows(rng, 7, 151936)
    for _ in range(2):
        check(sv, z1, 4, exclusions(rng, z1, 4), "bf16", ws)
        check(sv, z2, 8, None, "f32", ws)
    assert ws.read_error() == 0


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_topk_lanes_with_several_candidates(sv, dtype):
    """Rows where some 16-byte vectors hold a cluster of 2 to 8 equal high
    logits (one lane then marks several candidates in its chunk) and other
    chunks of the same row hold only scattered singles: the chunks of one call
    take the ballot count, the lane scan and, where more than 2K candidates
    gather, the exact merge.  Bit-exact against the oracle, ties by index."""
    rng = np.random.default_rng(5)
    R, V, K = 24, 40000, 4
    PV = 8 if dtype == "bf16" else 4
    z = rng.standard_normal((R, V)).astype(np.float32)
    for r in range(R):
        for j in rng.choice(V, 6, replace=False):
            z[r, j] = np.float32(6.0 + rng.random())
        for _ in range(int(rng.integers(1, 4))):
            v0 = int(rng.integers(0, V // PV)) * PV
            n = int(rng.integers(2, PV + 1))
            z[r, v0:v0 + n] = np.float32(6.5 if rng.random() < 0.5 else 7.5)
    check(sv, z, K, exclusions(rng, z, K), dtype)
    check(sv, z, K, None, dtype)


@pytest.mark.parametrize("dtype,K", [("bf16", 2), ("bf16", 4), ("bf16", 8), ("f32", 4)])
def test_topk_tiny_last_segment(sv, dtype, K):
    """Rows of 65552 bytes: two full 32 KB segments and a last segment of 16
    bytes (8 bf16 or 4 fp32 logits, one lane of one warp).  With 600 rows the
    streaming CTAs' chunk ranges start at every segment, so some warps meet a
    row first at its 16-byte tail: fewer than K lanes hold logits there, the
    bound the chunk starts from is -inf, and only the row's own elements may
    become candidates (the padding vectors read as -inf, and the shared memory
    behind them holds bytes of another chunk).  Half of the rows keep their
    largest logits in that tail, the other half their smallest."""
    rng = np.random.default_rng(17 + K)
    PV = 8 if dtype == "bf16" else 4
    V = 2 * (32768 // (2 if dtype == "bf16" else 4)) + PV
    R = 600
    z = rng.standard_normal((R, V)).astype(np.float32)
    z[0::2, V - PV:] = np.float32(9.0) + rng.random((R // 2, PV)).astype(np.float32)
    z[1::2, V - PV:] = np.float32(-9.0) - rng.random((R // 2, PV)).astype(np.float32)
    check(sv, z, K, exclusions(rng, z, K), dtype)
    check(sv, z, K, None, dtype)
