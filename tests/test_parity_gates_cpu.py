"""The parity comparison's whole-tensor gates bite at the DiT self-attention's magnitudes.

With Q and K scaled by 0.5 at D = 128 the scaled logits have std ~ 0.25, the softmax over
32760 keys is nearly uniform and |O| ~ 1 / sqrt(32760) ~ 0.005, far below the bf16 atol of
2e-2: the element-wise bound alone passes an all-zero O or one whose rows are shuffled.
The rel-L2 gate (the LingBot report's audit standard, rel-L2 <= 0.01 against FP64) and the
max|d| / max|ref| gate must reject both, and must still accept the oracle's own O rounded
to bf16 (what a correct kernel returns at best). CPU only: the oracle on 64 query rows.
"""

import numpy as np
import pytest
import torch

import oracle
from attention_sm_flash_gb300 import workloads
from gpu_util import GATE, TOL, compare


@pytest.fixture(scope="module")
def dit_rows():
    # the DiT self-attention's value recipe (Q, K 0.5 * N(0,1), V N(0,1), D 128, 32760
    # keys) on 64 query rows of one head
    w = workloads.small_case("gate", "gate_dit_rows", 1, 1, 1, 64, 32760, 128, "bf16", False,
                             seed=9001, has_bwd=False, qk_factor=0.5)
    inp = workloads.make_inputs(w)
    o_ref, _ = oracle.forward(inp["q"], inp["k"], inp["v"], w.scale, False, None)
    return o_ref


def test_magnitudes_are_below_atol(dit_rows):
    assert np.abs(dit_rows).max() < TOL["bf16"]["o"][0]
    assert np.sqrt(np.mean(dit_rows ** 2)) < 0.5 * TOL["bf16"]["o"][0]


def test_rounded_oracle_passes(dit_rows):
    got = torch.from_numpy(dit_rows).to(torch.bfloat16)
    compare("gate:o_bf16", got, dit_rows, *TOL["bf16"]["o"], gate=GATE["bf16"])


def test_elementwise_bound_alone_misses_zero_and_shuffled(dit_rows):
    # without the gates both wrong answers pass: the reason the gates exist
    compare("gate:zero_no_gate", torch.zeros(dit_rows.shape), dit_rows, *TOL["bf16"]["o"])
    perm = np.random.default_rng(3).permutation(dit_rows.shape[1])
    shuffled = torch.from_numpy(dit_rows[:, perm]).to(torch.bfloat16)
    compare("gate:shuffled_no_gate", shuffled, dit_rows, *TOL["bf16"]["o"])


def test_gates_reject_zero_output(dit_rows):
    with pytest.raises(AssertionError, match="rel-L2"):
        compare("gate:zero", torch.zeros(dit_rows.shape), dit_rows, *TOL["bf16"]["o"],
                gate=GATE["bf16"])


def test_gates_reject_row_shuffled_output(dit_rows):
    perm = np.random.default_rng(3).permutation(dit_rows.shape[1])
    shuffled = torch.from_numpy(dit_rows[:, perm]).to(torch.bfloat16)
    with pytest.raises(AssertionError, match="rel-L2|max"):
        compare("gate:shuffled", shuffled, dit_rows, *TOL["bf16"]["o"], gate=GATE["bf16"])


def test_gates_reject_one_wrong_row(dit_rows):
    # one query row replaced by another's: the max-ratio gate alone may catch what rel-L2
    # averages away over many rows; either gate failing is enough
    bad = dit_rows.copy()
    bad[0, 5] = dit_rows[0, 40]
    with pytest.raises(AssertionError):
        compare("gate:one_row", torch.from_numpy(bad), dit_rows, *TOL["bf16"]["o"],
                gate=GATE["bf16"])
