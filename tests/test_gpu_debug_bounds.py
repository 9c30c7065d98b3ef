"""The NVMOE_DEBUG_BOUNDS build (libnvfp4moe_debug.so, loaded with
NVMOE_LIBRARY=debug in a child process): in-kernel index checks record
NVMOE_ERR_DEVICE_BOUNDS and skip the access instead of touching memory out of
range.  The checks are provoked by declaring a bound smaller than the real
allocation, so every access the checks guard stays inside allocated memory
whatever the build does; on valid inputs the debug build gives the normal
library's bits."""
import json
import os
import subprocess
import sys

import pytest
import torch

pytestmark = pytest.mark.gpu
ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

CHILD = r'''
import json, sys, torch
sys.path.insert(0, ROOT)
from nvfp4_block_scaled_route_gb300 import binding as nb
from nvfp4_block_scaled_route_gb300 import synthetic as syn
assert nb.LIB_PATH.endswith("libnvfp4moe_debug.so")
DEV = "cuda"
out = {}

# 1. a forward on valid inputs: status 0, y saved for the parent
cfg = syn.CONFIGS["small"]
W1 = torch.stack([syn.draw_weight(cfg, 1, e, device=DEV) for e in range(cfg.E)])
W2 = torch.stack([syn.draw_weight(cfg, 2, e, device=DEV) for e in range(cfg.E)])
q1, s1, g1 = nb.quantize_weights(W1)
q2, s2, g2 = nb.quantize_weights(W2)
pw = nb.PreparedWeights.from_checkpoint(q1, s1, g1, q2, s2, g2)
layer = nb.MoELayer(pw, cfg.T, cfg.k, device=DEV)
ids, w = syn.draw_routing(cfg)
y = layer.forward(syn.draw_activations(cfg).to(DEV), ids.to(DEV), w.to(DEV),
                  taps={"path": nb.PATH_SEPARATE})
torch.cuda.synchronize()
out["forward_status"] = layer.status()
torch.save(y.cpu(), OUT)

# 2. scatter: 8 rows, slot_of 0..7, declared out_rows 4 (allocation: 8 rows)
H = 256
rows = torch.full((8, H // 2 + H // 16), 0x77, dtype=torch.uint8, device=DEV)
slot = torch.arange(8, dtype=torch.int32, device=DEV)
xq = torch.zeros((8, H // 2), dtype=torch.uint8, device=DEV)
xsf = torch.zeros(nb.sf_mma_bytes(8, H), dtype=torch.uint8, device=DEV)
st = torch.zeros(1, dtype=torch.int32, device=DEV)
nb.ep_scatter(rows, H, slot, 4, xq, xsf, status=st)
torch.cuda.synchronize()
out["scatter_status"] = int(st.item())
out["scatter_rows_written"] = int((xq.cpu() != 0).any(dim=1).sum())

# 3. gather: slot_out of 8 rows declared as 4 (a view of the first 4 rows)
src = torch.ones((8, H), dtype=torch.float16, device=DEV)
st.zero_()
g = nb.ep_gather(src[:4], slot, 8, status=st)
torch.cuda.synchronize()
out["gather_status"] = int(st.item())
out["gather_rows_nonzero"] = int((g.cpu() != 0).any(dim=1).sum())

# 4. quantiser: 8 token rows to rows 0..7, declared out_rows 4 (allocation 8)
x = torch.ones((8, H), dtype=torch.bfloat16, device=DEV)
q = torch.zeros((8, H // 2), dtype=torch.uint8, device=DEV)
ws = nb._workspace(nb.lib().nvfp4_quantize_workspace_size(8, H), DEV)
gs = torch.empty(1, dtype=torch.float32, device=DEV)
rc = nb.lib().nvfp4_quantize_act(nb._ptr(x), nb.BF16, 8, H, nb._ptr(slot), 1, 4, nb._ptr(q),
                                 None, None, nb._ptr(gs), nb._ptr(ws), ws.numel(), None)
torch.cuda.synchronize()
out["quant_rc"] = rc
out["quant_status"] = nb.read_status(ws)
out["quant_rows_written"] = int((q.cpu() != 0).any(dim=1).sum())
print("RESULT " + json.dumps(out))
'''


@pytest.fixture(scope="module")
def nb():
    import __graft_entry__
    __graft_entry__.build()
    from nvfp4_block_scaled_route_gb300 import binding
    return binding


def test_debug_bounds_build(nb, tmp_path):
    from nvfp4_block_scaled_route_gb300 import synthetic as syn
    out_file = str(tmp_path / "y_debug.pt")
    code = f"ROOT = {ROOT!r}\nOUT = {out_file!r}\n" + CHILD
    env = dict(os.environ, NVMOE_LIBRARY="debug")
    r = subprocess.run([sys.executable, "-c", code], env=env, capture_output=True, text=True,
                       timeout=600)
    assert r.returncode == 0, r.stdout[-2000:] + r.stderr[-2000:]
    line = [l for l in r.stdout.splitlines() if l.startswith("RESULT ")][-1]
    got = json.loads(line[len("RESULT "):])
    assert got["forward_status"] == 0
    assert got["scatter_status"] == 9 and got["scatter_rows_written"] == 4
    assert got["gather_status"] == 9 and got["gather_rows_nonzero"] == 4
    assert got["quant_rc"] == 0 and got["quant_status"] == 9 and got["quant_rows_written"] == 4
    # the same forward through the normal library: the same bits
    cfg = syn.CONFIGS["small"]
    W1 = torch.stack([syn.draw_weight(cfg, 1, e, device="cuda") for e in range(cfg.E)])
    W2 = torch.stack([syn.draw_weight(cfg, 2, e, device="cuda") for e in range(cfg.E)])
    q1, s1, g1 = nb.quantize_weights(W1)
    q2, s2, g2 = nb.quantize_weights(W2)
    pw = nb.PreparedWeights.from_checkpoint(q1, s1, g1, q2, s2, g2)
    layer = nb.MoELayer(pw, cfg.T, cfg.k, device="cuda")
    ids, w = syn.draw_routing(cfg)
    y = layer.forward(syn.draw_activations(cfg).to("cuda"), ids.to("cuda"), w.to("cuda"),
                      taps={"path": nb.PATH_SEPARATE}).cpu()
    assert torch.equal(y, torch.load(out_file))
