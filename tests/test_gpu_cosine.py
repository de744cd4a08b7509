"""GPU parity of the semantic fallback (AdaPLD section 3.2, Algorithm 1
SemanticFallback): cosine scores over a window of hidden states and the top
delta rows.  The GPU accumulates in fp32, so its scores may differ from the
fp64 oracle's by ~1e-6 (d = 4096): returned scores must lie within SCORE_TOL
of the oracle's score of the same row, and the returned rows must be the
oracle's except where two candidates' oracle scores are closer than TIE_TOL
(then either order is correct, and the GPU's choice must still be a valid
top-delta set: no excluded row may score more than TIE_TOL above an included
one)."""
import numpy as np
import pytest

import oracle
from speculative_decoding_verification_59_gb300 import workloads as W

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

SCORE_TOL = 1e-5
TIE_TOL = 2e-5


@pytest.fixture(scope="module")
def sv():
    import __graft_entry__
    __graft_entry__.build()
    import speculative_decoding_verification_59_gb300 as m
    return m


def dev(a, dtype=None):
    t = torch.from_numpy(np.ascontiguousarray(a)).cuda()
    return t.to(torch.bfloat16) if dtype == "bf16" else t


def check(sv, H, q, delta, dtype, positions=None):
    idx, pos, sc = sv.cosine_topk(dev(H, dtype), dev(q, dtype), delta,
                                  None if positions is None else dev(positions))
    torch.cuda.synchronize()
    idx, pos, sc = idx.cpu().numpy(), pos.cpu().numpy(), sc.cpu().numpy()
    ref = oracle.cosine_topk(H, q, delta, positions)
    S = ref["scores"]
    B, Wn = S.shape
    for b in range(B):
        got, want = idx[b], ref["idx"][b]
        n = min(delta, Wn)
        assert (got[n:] == -1).all() and (pos[b, n:] == -1).all()
        assert len(set(got[:n].tolist())) == n and (got[:n] >= 0).all()
        # scores of the returned rows
        assert np.all(np.abs(sc[b, :n] - S[b, got[:n]]) < SCORE_TOL), (b, sc[b], S[b, got[:n]])
        # same rows, except among oracle near-ties
        for k in range(n):
            if got[k] != want[k]:
                assert abs(S[b, got[k]] - S[b, want[k]]) < TIE_TOL, (b, k, got, want)
        excluded = np.setdiff1d(np.arange(Wn), got[:n])
        if excluded.size:
            assert S[b, excluded].max() < S[b, got[:n]].min() + TIE_TOL
        exp_pos = got[:n] if positions is None else positions[b, got[:n]]
        assert np.array_equal(pos[b, :n], exp_pos)
    return idx, ref


def test_cosine_full_workload(sv):
    c = W.make_cosine("cosine-b64")
    idx, ref = check(sv, c.hidden, c.query, c.delta, c.dtype, c.positions)
    # the planted near copies come out on top, in order of their noise
    assert (idx[0::2, :3] == ref["idx"][0::2, :3]).all()


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("W_,d,delta", [(1, 8, 1), (2, 8, 4), (33, 64, 3), (240, 2560, 8), (257, 4096, 4),
                                        (37, 2048, 4), (5, 16384, 2), (3, 1024, 8)])
def test_cosine_shapes(sv, dtype, W_, d, delta):
    """Window sizes from one row to more than a CTA's worth of rows, hidden
    sizes from one 16-byte vector to 32 KB (ragged batches of vectors)."""
    c = W.make_cosine("cosine-b64", B=5, W=W_, d=d, seed=W_ + d)
    H, q = c.hidden, c.query
    if dtype == "f32":
        rng = np.random.default_rng(d)
        H = rng.standard_normal(H.shape, dtype=np.float32)
        q = rng.standard_normal(q.shape, dtype=np.float32)
    check(sv, H, q, delta, dtype, None if W_ % 2 else c.positions)


@pytest.mark.parametrize("d", [128, 2048])
def test_cosine_zero_rows_and_ties(sv, d):
    """A short and a long hidden state (d = 2048 takes several batches of
    vectors per lane)."""
    rng = np.random.default_rng(11)
    B, Wn = 3, 40
    H = rng.standard_normal((B, Wn, d)).astype(np.float32)
    q = rng.standard_normal((B, d)).astype(np.float32)
    H[0, 5] = 0.0                      # zero row: score 0
    q[1] = 0.0                         # zero query: every score 0, rows in index order
    H[2, 7] = H[2, 30] = H[2, 12]      # exact ties: lower index first
    H[2, 12] = 2.0 * q[2]
    H[2, 7] = H[2, 30] = q[2]
    for dtype in ("f32", "bf16"):
        Hx, qx = (W.to_bf16_exact(H), W.to_bf16_exact(q)) if dtype == "bf16" else (H, q)
        idx, _ = check(sv, Hx, qx, 4, dtype)
        assert idx[1].tolist() == [0, 1, 2, 3]
        assert idx[2, :3].tolist() == [7, 12, 30]
