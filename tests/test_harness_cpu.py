"""The test harness's whole-output comparison, layer by layer, on the CPU:
pools holding the oracle's own whole-problem result pass it with no element
beyond 1 ulp, and planted faults (a wrong element, a write to an untargeted
slot, a row scattered to the wrong slot) fail it."""
import numpy as np
import pytest
import torch

import workloads as W
from tests import harness as Hn


def _with_oracle_result(spec):
    wl = W.make(spec, "cpu")
    h = Hn.snapshot(wl)
    ok, ov, _, _ = Hn.run_oracle(wl, h)
    before = wl.pool_k.clone() if wl.kind == "slide" else None
    wl.pool_k.view(torch.int16).copy_(torch.from_numpy(ok.view(np.int16)))
    if ov is not None:
        wl.pool_v.view(torch.int16).copy_(torch.from_numpy(ov.view(np.int16)))
    return wl, before


CASES = {
    "gqa": lambda: W.scaled(W.qwen_recall(), L=3, lens=(200, 65, 1)),
    "mla": lambda: W.scaled(W.dsv2_mla(), L=2, lens=(130, 7)),
    "slide": lambda: W.scaled(W.qwen_slide(), L=2, lens=(77, 40)),
}


@pytest.mark.parametrize("kind", list(CASES))
def test_layers_match_the_whole_problem(kind):
    wl, before = _with_oracle_result(CASES[kind]())
    st = Hn.check_layers(wl, range(wl.spec.L), kind, pool_before=before, workers=2)
    assert st and all(s.cancellation == 0 and s.max_ulp == 0 for s in st.values()), st
    assert sum(s.n for s in st.values()) > 0


@pytest.mark.parametrize("fault", ["element", "untouched", "swapped"])
def test_layers_catch_planted_faults(fault):
    wl, _ = _with_oracle_result(CASES["gqa"]())
    c = wl.chunks[0]
    k = wl.pool_k.view(torch.int16)
    if fault == "element":
        k[1, c.slots[5], 2, 17] += 3
    elif fault == "untouched":
        mask = torch.ones(wl.num_slots, dtype=torch.bool)
        for ch in wl.chunks:
            mask[ch.slots] = False
        k[0, torch.nonzero(mask)[0, 0], 0, 0] += 1
    else:
        a, b = c.slots[3], c.slots[4]
        ra, rb = k[2, a].clone(), k[2, b].clone()
        k[2, a], k[2, b] = rb, ra
    with pytest.raises(AssertionError):
        Hn.check_layers(wl, range(wl.spec.L), fault, workers=2)
