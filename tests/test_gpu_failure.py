"""Failure detection without a GPU fault: every pipeline wait in the kernels
is bounded, and a wait that runs out makes the kernel set MOE_DEV_TIMEOUT,
let its in-flight copies and MMAs finish, free its TMEM and return.

Each case runs a layer with a long K=14336 second GEMM (so that the
epilogue waits tens of microseconds for its accumulator) in a fresh process
whose wait limit is 1 ns, so a wait that is not satisfied within its first
few polls gives up: 512 rows (router and single-CTA grouped GEMM) and 4096
rows (the CTA-pair grouped GEMM, whose two CTAs count their loads on the
leader's barriers and settle the accounting of every stage in flight
before either exits). It checks that the status word reports the timeout,
that the CUDA context is still usable afterwards (a torch op and a second
layer call run), and that nothing raised."""
import json
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu
ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

CHILD = r"""
import json, sys
sys.path.insert(0, ROOT)
import torch
import top_routing_expert_gb300 as moe
import workloads as W
moe.build(); moe.load_library()
w = W.custom(TOKENS, 1024, 2, 1, 14336, 2.0, name="long_k")
inp = W.make_inputs(w, seed=0)
s = moe.MoeShape.make(w.T, w.H, w.E, w.k, w.h, w.cf)
ws = moe.Workspace(s)
d = {k: v.cuda() for k, v in inp.items() if v is not None}
y = torch.zeros((w.T, w.H), dtype=torch.bfloat16, device="cuda")
st = torch.zeros(1, dtype=torch.int32, device="cuda")
moe.moe_layer_fwd(s, d["x"], d["gate"], None, d["W1"], d["W2"], y, dev_status=st, ws=ws)
torch.cuda.synchronize()
first = int(st.item())
z = (torch.ones(1024, device="cuda") * 2).sum().item()
st2 = torch.zeros(1, dtype=torch.int32, device="cuda")
moe.moe_layer_fwd(s, d["x"], d["gate"], None, d["W1"], d["W2"], y, dev_status=st2, ws=ws)
torch.cuda.synchronize()
print(json.dumps({"first": first, "second": int(st2.item()), "torch_op": z}))
"""


@pytest.mark.parametrize("tokens", [512, 4096])
def test_wait_timeout_is_reported_and_context_survives(tokens):
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    env = dict(os.environ, MOE_GB300_WAIT_TIMEOUT_NS="1")
    code = CHILD.replace("ROOT", repr(ROOT)).replace("TOKENS", str(tokens))
    r = subprocess.run([sys.executable, "-c", code], env=env, capture_output=True, text=True,
                       timeout=300)
    assert r.returncode == 0, r.stderr[-2000:]
    out = json.loads(r.stdout.strip().splitlines()[-1])
    assert out["first"] & 8, out          # MOE_DEV_TIMEOUT
    assert out["torch_op"] == 2048.0      # the context is still usable
