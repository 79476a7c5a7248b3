"""First use of the library from several host threads at once (a fresh
process): the lazily fetched tensor-map encoder and the per-device launch
caches are set up by racing threads, and every launch must still succeed and
give the same bits as a launch from one thread."""
import os
import subprocess
import sys

import pytest
import torch

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

SCRIPT = r"""
import sys, threading
import torch
sys.path.insert(0, ROOT)
from compressed_kv_attention_compressplan_gb300 import ckv
from compressed_kv_attention_compressplan_gb300 import workloads as wl
ckv.load_library()
dev = torch.device("cuda")
w = wl.random_prefill(128, 512, torch.bfloat16, torch.float32, wl.COMPACT, [100, 0, 300], [600, 900, 257], seed=5,
                      num_requests_state=4)
plan_c, _, counts = ckv.plan_prefill(128, w.rid.to(dev), w.seq_lens.to(dev), w.extend_lens.to(dev), w.num_q_tokens)
torch.cuda.synchronize()
outs, errs = [None] * 4, []
barrier = threading.Barrier(4)

def run(i):
    try:
        s = torch.cuda.Stream()
        st, kv, ape = w.state.to(dev), w.kv_score.to(dev), w.ape.to(dev)
        torch.cuda.synchronize()
        barrier.wait()
        with torch.cuda.stream(s):
            outs[i] = ckv.compress_pool_prefill(128, 512, st, kv, ape, plan_c, counts, ckv.OUT_COMPACT, torch.float32,
                                                stream=s)
        s.synchronize()
    except Exception as e:
        errs.append(repr(e))

ts = [threading.Thread(target=run, args=(i,)) for i in range(4)]
[t.start() for t in ts]
[t.join() for t in ts]
assert not errs, errs
ref = ckv.compress_pool_prefill(128, 512, w.state.to(dev), w.kv_score.to(dev), w.ape.to(dev), plan_c, counts,
                                ckv.OUT_COMPACT, torch.float32)
torch.cuda.synchronize()
n = int(counts[0])
for o in outs:
    assert torch.equal(o[:n].view(torch.int32), ref[:n].view(torch.int32))
print("threads ok")
"""


def test_first_launches_from_several_threads():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from compressed_kv_attention_compressplan_gb300 import build as B

    B.build()
    r = subprocess.run([sys.executable, "-c", SCRIPT.replace("ROOT", repr(ROOT))], capture_output=True, text=True,
                       timeout=600)
    assert r.returncode == 0 and "threads ok" in r.stdout, r.stdout + r.stderr
