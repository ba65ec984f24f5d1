"""The roofline counts bench.py divides by, pinned to the formulas the pages print
(tests/golden/pages_constants.json, each entry with its citation)."""
import ast
import json
import os

import pytest

from linear_attention_serving_gb300 import roofline

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "pages_constants.json")


def _eval(formula, **names):
    """Evaluate a golden formula (numbers, names, + - * / **) with the given names."""
    tree = ast.parse(formula, mode="eval")
    allowed = (ast.Expression, ast.BinOp, ast.Add, ast.Sub, ast.Mult, ast.Div, ast.Pow, ast.Constant, ast.Name,
               ast.Load)
    for node in ast.walk(tree):
        assert isinstance(node, allowed), f"unexpected syntax in golden formula: {ast.dump(node)}"
    return eval(compile(tree, GOLDEN, "eval"), {"__builtins__": {}}, names)


@pytest.fixture(scope="module")
def golden():
    return json.load(open(GOLDEN))


@pytest.mark.parametrize("C,D", [(64, 128), (16, 64), (32, 256)])
def test_prefill_counts_follow_the_pages(golden, C, D):
    assert roofline.prefill_flops_per_chunk_head(C, D) == _eval(golden["flashkda_flops_per_chunk_head"]["formula"], C=C, D=D)
    assert roofline.prefill_bytes_per_chunk_head(C, D) == _eval(golden["flashkda_bytes_per_chunk_head"]["formula"], C=C, D=D)
    # the K1 / K2 split adds up to the pages' per-chunk total
    assert roofline.prep_bytes_per_chunk_head(C, D) + roofline.scan_bytes_per_chunk_head(C, D) == \
        roofline.prefill_bytes_per_chunk_head(C, D)


@pytest.mark.parametrize("T,H,n", [(8192, 16, 1), (32768, 32, 11), (1000, 3, 1)])
def test_kernel_level_bytes_follow_the_pages(golden, T, H, n):
    # per head the pages' kernel-level count; one state read and write per (sequence, head)
    per_head_one_seq = _eval(golden["flashkda_kernel_bytes"]["formula"], T=T, C=64, D=128)
    extra_states = (n - 1) * 8 * 128 ** 2
    assert roofline.prefill_kernel_bytes(T, H, n) == pytest.approx(H * (per_head_one_seq + extra_states), rel=1e-12)


def test_decode_counts_follow_the_pages(golden):
    for D in (64, 128):
        assert roofline.decode_flops_per_head_token(D) == _eval(golden["decode_flops_per_head_token"]["formula"], D=D)
        assert roofline.decode_bytes_per_head_token(D) == _eval(golden["decode_bytes_per_head_token"]["formula"], D=D)


def test_decode_step_bytes_are_dominated_by_the_state():
    """The MTP step's count: the fp32 state once in and once out is the pages' 8 D^2
    per (sequence, head); inputs, cache and outputs come on top, and the fused step
    adds the convolution state, the output gates and the replayed q."""
    N, H, W, acc = 256, 96, 5, 512
    plain = roofline.decode_step_bytes(N, H, W, acc)
    fused = roofline.decode_fused_step_bytes(N, H, W, acc)
    state = N * H * roofline.decode_bytes_per_head_token()
    assert state < plain < 1.25 * state
    conv_state_in_out = N * H * 2 * 9 * 128 * 4
    assert plain + conv_state_in_out < fused < 1.1 * plain
    # more accepted drafts replay more cached inputs
    assert roofline.decode_step_bytes(N, H, W, 2 * acc) > plain
