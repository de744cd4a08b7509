"""Several host threads drive the library at once, each on its own CUDA stream
with its own workspace and inputs: every call's outputs must equal those of
the same call made alone.  The scenario runs in a fresh process, so the
threads are the first users of the library's host-side state (the
per-device caches of device properties, shared-memory opt-ins and
occupancy), and it checks that calls sharing no workspace are independent."""
import os
import subprocess
import sys
import threading

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

pytestmark = pytest.mark.gpu


def _dev(torch, a, dtype=None):
    t = torch.from_numpy(np.ascontiguousarray(a)).cuda()
    return t.to(torch.bfloat16) if dtype == "bf16" else t


def _job(sv, W, torch, seed):
    """Inputs of one thread and a function that runs its calls on a stream."""
    name = ("chain-b8", "chain-b64", "chain-b256")[seed % 3]
    x = W.make_chain(name, B=6, gamma=3 + seed % 4, V=(4096, 8192, 20000)[seed % 3], seed=100 + seed)
    t = W.make_tree(B=3, V=4096, seed=200 + seed)
    zt, zd = _dev(torch, x.target, x.dtype), _dev(torch, x.draft, x.dtype)
    xt, u = _dev(torch, x.draft_tokens), _dev(torch, x.uniforms)
    tt = _dev(torch, t.target, "bf16")
    tn, tp = _dev(torch, t.node_tokens), _dev(torch, t.parents)

    def run(stream, reps):
        ws = sv.Workspace()
        out = []
        with torch.cuda.stream(stream):
            for _ in range(reps):
                out.append([
                    *sv.verify_sample(zt, zd, xt, u, x.T, logprobs=True, workspace=ws, stream=stream),
                    *sv.verify_sample(zt, zd, xt, u, x.T, workspace=ws, stream=stream, lazy=True),
                    *sv.verify_greedy(zt, xt, workspace=ws, stream=stream),
                    *sv.verify_tree_greedy(tt, tn, tp, workspace=ws, stream=stream)])
            stream.synchronize()
        return [[a.cpu().numpy() for a in r] for r in out]

    return run


def scenario(n=6, reps=3):
    """Runs the threads, then each job alone, and compares; returns a list of
    mismatches and errors (empty: pass)."""
    import torch

    import speculative_decoding_verification_59_gb300 as sv
    from speculative_decoding_verification_59_gb300 import workloads as W

    jobs = [_job(sv, W, torch, s) for s in range(n)]
    torch.cuda.synchronize()                         # inputs made on the default stream
    results, problems = [None] * n, []

    def worker(i):
        try:
            results[i] = jobs[i](torch.cuda.Stream(), reps)
        except Exception as e:                       # reported by the caller
            problems.append(("error", i, repr(e)))

    threads = [threading.Thread(target=worker, args=(i,)) for i in range(n)]
    for th in threads:
        th.start()
    for th in threads:
        th.join()
    for i in range(n):
        alone = jobs[i](torch.cuda.Stream(), 1)[0]
        for rep in results[i] or []:
            for k, (got, want) in enumerate(zip(rep, alone)):
                if not np.array_equal(got, want, equal_nan=True):
                    problems.append(("mismatch", i, k))
    return problems


def test_concurrent_host_threads_match_single_threaded():
    import __graft_entry__
    __graft_entry__.build()
    env = dict(os.environ, PYTHONPATH=ROOT + os.pathsep + os.environ.get("PYTHONPATH", ""))
    r = subprocess.run([sys.executable, os.path.abspath(__file__)], cwd=ROOT, env=env,
                       capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stdout[-2000:] + r.stderr[-2000:]
    assert "threads ok" in r.stdout


if __name__ == "__main__":
    found = scenario()
    print(found if found else "threads ok")
    sys.exit(1 if found else 0)
