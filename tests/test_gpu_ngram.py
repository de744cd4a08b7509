"""GPU parity of lexical (n-gram) retrieval (AdaPLD sections 3.2-3.3,
Algorithm 1 LexicalRetrieval and d_main) against the oracle: match counts,
ordered match lists and drafts are integers and must be identical."""
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


def check(sv, tokens, lengths, w, L, cap, ws=None):
    t = torch.from_numpy(np.ascontiguousarray(tokens, dtype=np.int32)).cuda()
    n = torch.from_numpy(np.ascontiguousarray(lengths, dtype=np.int32)).cuda()
    cnt, mat, dr = sv.ngram_retrieve(t, n, w, L, cap, workspace=ws)
    torch.cuda.synchronize()
    ref = oracle.ngram_retrieve(tokens, lengths, w, L, cap)
    assert np.array_equal(cnt.cpu().numpy(), ref["count"])
    assert np.array_equal(mat.cpu().numpy(), ref["matches"])
    assert np.array_equal(dr.cpu().numpy(), ref["draft"])
    return ref


@pytest.mark.parametrize("w", [1, 2, 3, 4, 5, 6, 7, 8])
@pytest.mark.parametrize("n_max", [4, 1024, 5000, 70000, 300000])
def test_ngram_small_alphabet(sv, w, n_max):
    """Every window length (each has its own kernel), contexts from one
    16-byte vector to more than 64 tiles of 4096 positions (segments of two
    tiles), over a 3-token alphabet: matches nearly everywhere."""
    if n_max % 4:
        n_max += 4 - n_max % 4
    rng = np.random.default_rng(w * 1000 + n_max)
    B = 12
    t = rng.integers(0, 3, size=(B, n_max)).astype(np.int32)      # dense matches
    lengths = rng.integers(1, n_max + 1, size=B).astype(np.int32)
    lengths[0] = 1
    lengths[1] = min(w, n_max)
    lengths[2] = n_max
    for cap in (1, 5, 300):
        check(sv, t, lengths, w, 9, cap)


def test_ngram_full_size_workload(sv):
    g = W.make_ngram("ngram-b64")
    ref = check(sv, g.tokens, g.lengths, g.w, g.L, g.max_matches)
    assert (ref["count"] > 0).sum() >= g.tokens.shape[0] // 2       # hits and misses both present
    assert (ref["count"] == 0).any()


def test_ngram_bad_lengths_and_no_draft(sv):
    g = W.make_ngram("ngram-b64", B=6, n_max=4096, n_min=1024)
    lengths = g.lengths.copy()
    lengths[1] = 0
    lengths[4] = 4097
    ws = sv.Workspace()
    t = torch.from_numpy(g.tokens).cuda()
    n = torch.from_numpy(lengths).cuda()
    cnt, mat, dr = sv.ngram_retrieve(t, n, 3, 0, 16, workspace=ws)
    torch.cuda.synchronize()
    c = cnt.cpu().numpy()
    assert c[1] == -1 and c[4] == -1 and (mat.cpu().numpy()[[1, 4]] == -1).all()
    assert ws.read_error() & sv.SPEC_DEVERR_TOKEN_RANGE
    ok = [0, 2, 3, 5]
    ref = oracle.ngram_retrieve(g.tokens[ok], g.lengths[ok], 3, 0, 16)
    assert np.array_equal(c[ok], ref["count"])
    assert np.array_equal(mat.cpu().numpy()[ok], ref["matches"])
