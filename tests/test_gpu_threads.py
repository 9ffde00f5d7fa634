"""Calls from several host threads at once.  include/usp.h promises that the
calls keep no state and may be issued from any host thread, with the
library's per-process lookups (the tensor-map encoder, the status word's
address, the SM count) race-free.  A fresh child process makes its first
calls from four threads at the same time, each on its own stream and
problem; every thread's results must be bitwise those of the same problem
run alone afterwards (the two-pass backward is deterministic)."""
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

CHILD = r'''
import threading, sys
import torch
sys.path.insert(0, "tests")
from ulysses_sequence_attention_usp_gb300.pipeline import UlyssesAttention
from gpu_util import to_dev
from test_gpu_attention import _setup

CASES = [(1000, 2, 8, 2, 128, None), (777, 4, 8, 4, 64, [100, 1, 300, 376]),
         (600, 2, 16, 2, 128, [200, 400]), (300, 2, 8, 2, 128, [100, 0, 150, 0, 50])]
setups = [_setup(c, seed=20 + i) for i, c in enumerate(CASES)]
inputs = [[to_dev(x) for x in (inp.q, inp.k, inp.v, inp.do)] for _, inp in setups]
torch.cuda.synchronize()
results, errors = [None] * len(CASES), []
barrier = threading.Barrier(len(CASES))

def make(i):
    wl, inp = setups[i]
    return UlyssesAttention(wl.S, wl.P, wl.Hq, wl.Hkv, wl.D, cu_seqlens=inp.cu,
                            rope_base=wl.rope_base)

def outs(ua):
    return [t.clone() for t in (ua.o, ua.lse, ua.dq, ua.dk, ua.dv)]

def work(i):
    try:
        s = torch.cuda.Stream()
        with torch.cuda.stream(s):
            ua = make(i)
            barrier.wait()                 # first calls from all threads together
            for _ in range(4):
                ua.step(*inputs[i])
            res = outs(ua)
            s.synchronize()
        results[i] = res
    except Exception as e:                 # reported by the main thread
        errors.append(repr(e))

threads = [threading.Thread(target=work, args=(i,)) for i in range(len(CASES))]
for t in threads:
    t.start()
for t in threads:
    t.join()
assert not errors, errors
torch.cuda.synchronize()
for i in range(len(CASES)):
    ua = make(i)
    ua.step(*inputs[i])
    ua.check()
    for a, b in zip(outs(ua), results[i]):
        if a.dtype == torch.bfloat16:
            a, b = a.view(torch.int16), b.view(torch.int16)
        assert torch.equal(a, b), i
print("threads ok")
'''


def test_first_calls_from_four_threads_match_serial_runs():
    r = subprocess.run([sys.executable, "-c", CHILD], cwd=ROOT, capture_output=True, text=True,
                       timeout=600)
    assert r.returncode == 0 and "threads ok" in r.stdout, r.stdout[-3000:] + r.stderr[-3000:]
