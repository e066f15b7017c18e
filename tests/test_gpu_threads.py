"""Two host threads driving one device at once.

The library keeps per-device launch state (the SM count, each kernel's
shared-memory limit, the fused write's wave size) in caches that the first
call on a device fills.  Calls from several host threads may race to fill
them; each must still launch correctly.  The race needs a process in which
no call has run yet, so the test runs in a child process: two threads wait
at a barrier, then each makes its first decode calls (both stage-1 kernels,
the merge and the fused write) on its own stream, and the results are
compared with the oracle.
"""
import os
import subprocess
import sys
import textwrap

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

CHILD = textwrap.dedent(r"""
    import sys, threading
    sys.path.insert(0, sys.argv[1])
    sys.path.insert(0, sys.argv[1] + "/tests")
    import numpy as np, torch
    import mla_paged_kv_concat_gb300 as mla
    from mla_paged_kv_concat_gb300 import workloads as W
    from _helpers import Dev, assert_close, oracle_cache, oracle_decode, unit_pairs

    mla.load()
    torch.cuda.init()
    cases = [W.make_workload("thr16", seed=301, seq_lens=[700, 1300, 64, 2000], num_heads=16),
             W.make_workload("thr128", seed=302, seq_lens=[900, 3000], num_heads=128)]
    devs = [Dev(w) for w in cases]
    outs = [None, None]
    errors = []
    go = threading.Barrier(2)

    def work(i):
        try:
            w, d = cases[i], devs[i]
            s = torch.cuda.Stream()
            with torch.cuda.stream(s):
                go.wait()
                d.write()
                o, lse = d.decode(mla.mla_num_kv_splits(w.max_seq_len, 152))
                o1, lse1 = d.decode(1)
            s.synchronize()
            outs[i] = (o, lse, o1, lse1)
        except Exception as e:  # reported by the main thread
            errors.append(repr(e))

    th = [threading.Thread(target=work, args=(i,)) for i in range(2)]
    for t in th:
        t.start()
    for t in th:
        t.join()
    assert not errors, errors
    for w, d, (o, lse, o1, lse1) in zip(cases, devs, outs):
        cache = oracle_cache(w)
        assert d.cache_numpy().tobytes() == cache.tobytes()
        pairs = unit_pairs(w, 128, extra=32, seed=5)
        o_ref, lse_ref = oracle_decode(w, cache, pairs=pairs)
        assert_close(o, lse, o_ref, lse_ref, pairs=pairs, what=w.name)
        assert_close(o1, lse1, o_ref, lse_ref, pairs=pairs, what=w.name + " S=1")
        assert int(d.err.item()) == 0
    print("threads ok")
""")


def test_two_host_threads_first_calls_on_one_device(cuda_dev):
    r = subprocess.run([sys.executable, "-c", CHILD, ROOT], capture_output=True, text=True,
                       timeout=600)
    assert r.returncode == 0, r.stdout[-2000:] + r.stderr[-4000:]
    assert "threads ok" in r.stdout
