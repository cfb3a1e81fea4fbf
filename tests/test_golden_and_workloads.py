"""CPU tests of the work accounting (against the pages' printed figures) and of the
seeded input generators."""

import json
import os

import numpy as np
import torch

from attention_sm_flash_gb300 import metrics, workloads

HERE = os.path.dirname(os.path.abspath(__file__))


def test_utilisation_rule_reproduces_printed_percentages():
    with open(os.path.join(HERE, "golden", "page_utilisation.json")) as f:
        gold = json.load(f)
    peak = gold["peak_tflops"] * 1e12
    for c in gold["cases"]:
        fl = metrics.fwd_flops(c["B"], c["H"], c["H"], c["Q"], c["K"], c["D"], False)
        pct = 100.0 * metrics.utilisation(fl, c["time_ms"] * 1e-3, peak)
        assert abs(pct - c["printed_pct"]) <= 0.05, (c["what"], pct)


def test_visible_pairs_closed_forms():
    # non-causal: Sq * L per head; causal square: S (S + 1) / 2 per head
    assert metrics.visible_pairs(2, 4, 2, 7, 9, False) == 2 * 4 * 7 * 9
    assert metrics.visible_pairs(1, 3, 3, 10, 10, True) == 3 * 55
    lens = np.array([[5, 0]])
    assert metrics.visible_pairs(1, 4, 2, 3, 6, False, lens) == 2 * 3 * 5
    # bottom-right causal, Sq = 3, L = 5: rows see 3, 4, 5 keys
    assert metrics.visible_pairs(1, 1, 1, 3, 5, True) == 12
    # brute force on a random small case
    rng = np.random.default_rng(0)
    lens = rng.integers(0, 8, size=(2, 2))
    want = 0
    for b in range(2):
        for h in range(4):
            L = lens[b, h // 2]
            for i in range(6):
                want += sum(1 for j in range(L) if j <= i + L - 6)
    assert metrics.visible_pairs(2, 4, 2, 6, 7, True, lens) == want


def test_workload_shapes_and_flops():
    w = workloads.get("c4")
    assert (w.B, w.Hq, w.Sq, w.Skv, w.D) == (1, 40, 32760, 32760, 128)
    assert 32760 == 21 * 30 * 52
    assert abs(metrics.fwd_flops(1, 40, 40, 32760, 32760, 128, False) - 2.198e13) < 1e10
    w2 = workloads.get("c2")
    f2 = metrics.fwd_flops(w2.B, w2.Hq, w2.Hkv, w2.Sq, w2.Skv, w2.D, True)
    assert f2 == 4 * 64 * 8 * 12 * 1024 * 1025 / 2


def test_small_inputs_are_seeded_and_rounded():
    w = workloads.small_case("t", "t", 2, 4, 2, 33, 47, 64, "bf16", True, 99,
                             lens_kind="per_head_uniform", lens_lo=1, lens_hi=47)
    a = workloads.make_inputs(w)
    b = workloads.make_inputs(w)
    for key in ("q", "k", "v", "do", "kv_lens"):
        assert torch.equal(a[key], b[key])
    assert a["q"].dtype == torch.bfloat16 and a["q"].shape == (2, 33, 4, 64)
    assert a["k"].shape == (2, 47, 2, 64) and a["kv_lens"].dtype == torch.int32
    assert int(a["kv_lens"].min()) >= 1 and int(a["kv_lens"].max()) <= 47
    # values are the RNE rounding of the fp32 draws, in the order Q, K, V, dO
    g = torch.Generator().manual_seed(99)
    q32 = torch.randn((2, 33, 4, 64), generator=g)
    assert torch.equal(q32.to(torch.bfloat16), a["q"])
    c = workloads.make_inputs(workloads.small_case("t", "t", 2, 4, 2, 33, 47, 64, "bf16",
                                                   True, 100))
    assert not torch.equal(a["q"], c["q"])


def test_cross_attention_lengths():
    w = workloads.get("c5")
    assert w.lens_kind == "fixed" and w.lens_fixed == 300 and w.Skv == 512
