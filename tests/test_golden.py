"""Checks of the oracle against the hand-derived worked examples and the
page facts stored under tests/golden/ (each entry carries its source)."""
import json
import os

import numpy as np
import torch

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _load(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


def _bits(x):
    return x.view(torch.int16).numpy().view(np.uint16)


def test_hand_examples_1x32(orc):
    ex = _load("hand_examples.json")
    for case in ex["groups_1x32"]:
        x = torch.zeros(1, 32, dtype=torch.bfloat16)
        for i, v in case["values"].items():
            x[0, int(i)] = float(v)
            assert float(x[0, int(i)]) == float(v)       # exactly representable
        q, s = orc.quant_rows(_bits(x))
        assert s[0, 0] == case["scale_code"], case["why"]
        for i, code in case["payload"].items():
            assert q[0, int(i)] == int(code, 16), case["why"]


def test_hand_example_32x32(orc):
    t = _load("hand_examples.json")["tile_32x32"]
    w = torch.zeros(32, 32, dtype=torch.bfloat16)
    for rc, v in t["values"].items():
        r, c = map(int, rc.split(","))
        w[r, c] = float(v)
    q, s_fwd, s_bwd = orc.quant_32x32(_bits(w))
    assert np.all(s_fwd == t["tile_scale_code"]) and np.all(s_bwd == t["tile_scale_code"])
    for rc, code in t["payload"].items():
        r, c = map(int, rc.split(","))
        assert q[r, c] == int(code, 16), t["why"]
    q1, s1 = orc.quant_rows(_bits(w))
    assert s1[5, 0] == t["row5_1x32_scale_code"] and q1[5, 3] == int(t["row5_1x32_payload_col3"], 16)


def test_page_facts_tensor_counts_and_bytes(orc):
    f = _load("page_facts.json")
    assert f["elements_per_scale"]["value"] == 32
    w = torch.randn(64, 96).to(torch.bfloat16)
    dual = orc.quant_dual(_bits(w))                        # mxfp8: fwd + bwd copies
    blk = orc.quant_32x32(_bits(w))                        # mxfp8-32x32: one payload
    assert len(dual) == f["allgather_tensor_count"]["value"]["mxfp8"]
    assert len(blk) == f["allgather_tensor_count"]["value"]["mxfp8-32x32"]
    # one scale per 32 elements in every scale tensor
    for q, s in ((dual[0], dual[1]), (dual[2], dual[3]), (blk[0], blk[1])):
        assert s.size * 32 == q.size
    assert blk[2].size * 32 == blk[0].size
    # the 32x32 form gathers one payload instead of two
    assert sum(a.nbytes for a in blk) == sum(a.nbytes for a in dual) - w.numel()
