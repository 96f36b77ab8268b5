"""Calls from several host threads at once, each on its own stream and workspace (the C ABI
allows that), including the first calls of a process, which set up each kernel's shared-memory
limit and the device's SM count under a lock. Run in a fresh process so that those first calls
really race. Each thread's results must equal a sequential rerun: the forward's output and
LSE and the backward's dK and dV bitwise, dQ within 1e-6 of its largest magnitude (its
partial sums arrive in any order)."""
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

SCRIPT = r'''
import sys, threading
sys.path.insert(0, ROOT)
import torch
from tests.gpu_util import Problem
from ulysses_sequence_seq_gb300.synth import custom_workload, head_sharded_bits

shapes = [([300, 129, 1, 270], 4, 2, 128), ([700, 64], 2, 2, 64), ([513, 200], 8, 1, 128), ([1000], 2, 1, 64)]
probs = []
for n, (lens, hq, hkv, D) in enumerate(shapes):
    w = custom_workload("threads%d" % n, lens, sp=1, hq=hq, hkv=hkv, head_dim=D, index=60 + n)
    q, k, v, do = (head_sharded_bits(w, t) for t in ("q", "k", "v", "do"))
    probs.append(Problem(q, k, v, w.cu_seqlens(), True, do_bits=do))
torch.cuda.synchronize()

def run(p):
    o, lse, st = p.forward()
    dq, dk, dv, st2 = p.backward(o, lse, torch.float32)
    torch.cuda.current_stream().synchronize()
    return [x.clone() for x in (o, lse, dq, dk, dv)], (st, st2)

results = [None] * len(probs)
errors = []
start = threading.Barrier(len(probs))

def work(i):
    try:
        s = torch.cuda.Stream()
        with torch.cuda.stream(s):
            start.wait()
            for _ in range(3):
                results[i] = run(probs[i])
    except Exception as e:
        errors.append(repr(e))

threads = [threading.Thread(target=work, args=(i,)) for i in range(len(probs))]
for t in threads:
    t.start()
for t in threads:
    t.join()
assert not errors, errors
for i, p in enumerate(probs):
    got, st = results[i]
    assert st == (0, 0), st
    want, st2 = run(p)
    assert st2 == (0, 0)
    o, lse, dq, dk, dv = got
    wo, wl, wq, wk, wv = want
    assert torch.equal(o.view(torch.int16), wo.view(torch.int16)) and torch.equal(lse, wl)
    assert torch.equal(dk.view(torch.int32), wk.view(torch.int32)) and torch.equal(dv.view(torch.int32), wv.view(torch.int32))
    assert float((dq - wq).abs().max()) <= 1e-6 * float(wq.abs().max())
print("threads ok")
'''


def test_concurrent_calls_from_host_threads():
    from tests.gpu_util import needs_gpu
    needs_gpu()
    out = subprocess.run([sys.executable, "-c", SCRIPT.replace("ROOT", repr(ROOT), 1)], capture_output=True,
                         text=True, timeout=600, cwd=ROOT)
    assert out.returncode == 0 and "threads ok" in out.stdout, out.stdout[-2000:] + out.stderr[-4000:]
