"""ATTN_LOG=1: one stderr line per forward / backward call naming the chosen
schedule (the library reads the variable once, so this runs in a child)."""
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

CHILD = r"""
import torch, attn_inputs, online_softmax_attention_gb300 as attn
x = attn_inputs.make(dtype="bf16", H=2, D=128, seed=3, n_q=300, backward=True)
q, k, v, dO = (x[n].cuda() for n in ("q", "k", "v", "dO"))
o, lse = attn.fwd(q, k, v, causal=True, num_splits=2)
attn.bwd(q, k, v, o, lse, dO, causal=True)
torch.cuda.synchronize()
"""


def test_log_lines_name_the_schedule():
    env = dict(os.environ, ATTN_LOG="1", PYTHONPATH=ROOT)
    r = subprocess.run([sys.executable, "-c", CHILD], cwd=ROOT, env=env, capture_output=True,
                       text=True, timeout=300)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stderr.splitlines() if ln.startswith("[attn]")]
    assert any("fwd n_q=300" in ln and "kernel=tc" in ln and "splits=2" in ln for ln in lines), lines
    assert any("bwd n_q=300" in ln and "dq=separate" in ln for ln in lines), lines
    env.pop("ATTN_LOG")
    r = subprocess.run([sys.executable, "-c", CHILD], cwd=ROOT, env=env, capture_output=True,
                       text=True, timeout=300)
    assert r.returncode == 0 and "[attn]" not in r.stderr
