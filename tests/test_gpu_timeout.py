"""The bounded waits of the tensor-core kernels, made to run out.

Every pipeline wait of relocate_patch_umma_kernel and patch_form_kernel gives
up after a bound (1 s; the environment variable KAMERA_WAIT_LIMIT_NS, read at
each call, overrides it).  Relocation: KAMERA_TEST_WITHHOLD_LOADS=1 makes the
producer issue no loads, so the other roles' first waits cannot be met and
run out after the bound (here 1 ms).  Patch formation: with a bound of 0 the
first poll that finds a wait unmet gives up.  Either way the call must still
return, report KAMERA_DEVERR_TIMEOUT, and leave the device usable -- each CTA
drained its own loads, copies and MMAs and released its tensor memory --
which a normal call right after, on the same stream, shows by matching the
oracle (a CTA that kept its tensor memory would leave the next launch's
allocation waiting).  Nothing here faults: every address stays valid and
every wait is bounded."""
import numpy as np
import pytest
import torch

import oracle as O
import position_invariant_kv_chunk_gb300 as K
import workloads as W
from tests import harness as Hn

pytestmark = pytest.mark.gpu
DEV = "cuda"
TIMEOUT = 32   # KAMERA_DEVERR_TIMEOUT


@pytest.mark.parametrize("name", ["qwen_recall", "dsv2_mla"])
def test_relocate_wait_runs_out_then_recovers(name, monkeypatch):
    spec = W.scaled(W.CONFIGS[name](), L=3, lens=(1296, 200, 65, 900))
    wl = W.make(spec, DEV)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    monkeypatch.setenv("KAMERA_WAIT_LIMIT_NS", "1000000")
    monkeypatch.setenv("KAMERA_TEST_WITHHOLD_LOADS", "1")
    Hn.run_gpu(wl, err=err)
    torch.cuda.synchronize()
    assert int(err.item()) & TIMEOUT, f"no wait ran out (d_err = {int(err.item())})"
    monkeypatch.delenv("KAMERA_WAIT_LIMIT_NS")
    monkeypatch.delenv("KAMERA_TEST_WITHHOLD_LOADS")
    again = W.make(spec, DEV)
    h = Hn.snapshot(again)
    err2 = torch.zeros(1, dtype=torch.int32, device=DEV)
    Hn.run_gpu(again, err=err2)
    Hn.check_parity(again, h, f"{name} after a timed-out call")
    assert int(err2.item()) == 0


def test_patch_form_wait_runs_out_then_recovers(monkeypatch):
    spec = W.DeficitSpec("timeout_pf", L=2, length=700, H=2, d=128, m=16, kv=1)
    x = W.make_deficit(spec, DEV)
    xb = x.reshape(spec.L, spec.length, spec.H, spec.d).permute(0, 2, 1, 3)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    monkeypatch.setenv("KAMERA_WAIT_LIMIT_NS", "0")
    K.kamera_form_patch(xb, spec.m, err=err)
    torch.cuda.synchronize()
    assert int(err.item()) & TIMEOUT, f"no wait ran out (d_err = {int(err.item())})"
    monkeypatch.delenv("KAMERA_WAIT_LIMIT_NS")
    err2 = torch.zeros(1, dtype=torch.int32, device=DEV)
    u, v = K.kamera_form_patch(xb, spec.m, err=err2)
    torch.cuda.synchronize()
    assert int(err2.item()) == 0
    for o in range(spec.L):
        for i in range(spec.H):
            blk = xb[o, i].float().cpu().numpy().astype(np.float64)
            uo, vo = O.form_patch(blk, spec.m)
            rec = u[o, i].float().cpu().numpy().astype(np.float64) @ v[o, i].float().cpu().numpy().astype(np.float64).T
            ref = uo @ vo.T
            assert np.linalg.norm(rec - ref) <= 8e-3 * np.linalg.norm(ref)

