"""The oracle against hand-worked cases stored under tests/golden/ (no GPU needed).

Each fixture states the passage of the pages the operation follows and derives its
expected values by hand from the definitions: exact integers (E4M3 codes, scale bytes,
expert indices, counts) and closed-form expressions for real values, evaluated here with
Python's math functions only.
"""
import math
import os

import numpy as np
import pytest

from oracle import moe_oracle as om
from oracle import mx

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
MATH = {"e": math.e, "pi": math.pi, "log": math.log, "exp": math.exp, "sqrt": math.sqrt}


def _expr(text, names=None):
    return eval(text, {"__builtins__": {}}, {**MATH, **(names or {})})  # noqa: S307 (fixture arithmetic)


def _lines(name):
    for raw in open(os.path.join(GOLDEN, name)):
        line = raw.strip()
        if line and not line.startswith("#"):
            yield line


def _mx_cases(name="mx_blocks.txt"):
    cases, cur = [], None
    for line in _lines(name):
        key, _, rest = line.partition(" ")
        if key == "case":
            cur = {"name": rest, "values": np.zeros(32), "codes": np.zeros(32, np.uint8)}
            cases.append(cur)
        elif key == "values":
            for item in rest.split():
                i, v = item.split(":")
                cur["values"][int(i)] = float.fromhex(v) if "0x" in v else float(v)
        elif key == "scale":
            cur["scale"] = int(rest)
        elif key == "codes":
            for item in rest.split():
                i, c = item.split(":")
                cur["codes"][int(i)] = int(c, 16)
    return cases


@pytest.mark.parametrize("case", _mx_cases(), ids=lambda c: c["name"])
def test_mx_block_by_hand(case):
    codes, scales = mx.mx_quantize(case["values"].reshape(1, 32))
    assert int(scales[0, 0]) == case["scale"]
    assert np.array_equal(codes[0], case["codes"]), [hex(c) for c in codes[0]]


@pytest.mark.parametrize("case", _mx_cases("mx4_blocks.txt"), ids=lambda c: c["name"])
def test_mx4_block_by_hand(case):
    codes, scales = mx.mx4_quantize(case["values"].reshape(1, 32))
    assert int(scales[0, 0]) == case["scale"]
    assert np.array_equal(codes[0], case["codes"]), [hex(c) for c in codes[0]]


def _routing_blocks():
    blocks, cur = [], None
    for line in _lines("routing.txt"):
        key, _, rest = line.partition(" ")
        if key == "score":
            f = rest.split()
            cur = {"score": f[0], "k": int(f[2]), "E": int(f[4]), "logits": [], "idx": [], "w": []}
            blocks.append(cur)
        elif key == "token":
            lg, _, out = rest.partition("->")
            idx, _, w = out.partition("|")
            cur["logits"].append([_expr(t) for t in lg.split()])
            cur["idx"].append([int(t) for t in idx.split()])
            cur["w"].append([_expr(t) for t in w.split()])
        elif key == "split_sizes":
            cur["split"] = [int(t) for t in rest.split()]
    return blocks


@pytest.mark.parametrize("block", _routing_blocks(), ids=lambda b: b["score"])
def test_routing_by_hand(block):
    score = om.SOFTMAX if block["score"] == "softmax" else om.SIGMOID
    logits = np.array(block["logits"], np.float32)
    idx, w = om.route(logits, block["k"], score, np.float64)
    assert np.array_equal(idx, np.array(block["idx"]))
    np.testing.assert_allclose(w, np.array(block["w"]), rtol=0, atol=1e-7)  # fp32 logits
    split, offsets, _, _ = om.dispatch(idx, block["E"])
    assert list(split) == block["split"]
    assert list(offsets) == list(np.concatenate([[0], np.cumsum(block["split"])])[: len(offsets)])


def test_swiglu_one_token_by_hand():
    names = {}
    for line in _lines("swiglu_one_token.txt"):
        key, _, expr = line.partition("=")
        names[key.strip()] = _expr(expr.strip(), names)
    x = np.array([names["x"]], np.float64)
    logits = np.array([names["logits"]], np.float64)
    dy = np.array([names["dy"]], np.float64)
    w_gu = np.array([names["w_gu0"], names["w_gu1"]], np.float64)
    w_d = np.array([names["w_d0"], names["w_d1"]], np.float64)
    fwd = om.moe_forward(x, logits, w_gu, w_d, 2, om.SOFTMAX)
    bwd = om.moe_backward(x, logits, w_gu, w_d, dy, fwd, 2, om.SOFTMAX)
    close = lambda a, b: np.testing.assert_allclose(np.asarray(a, np.float64), np.asarray(b), rtol=1e-12, atol=1e-14)  # noqa: E731
    close(fwd["Y"][0], names["Y"])
    close(bwd["dX"][0], names["dX"])
    close(bwd["dW_gu"][0], names["dW_gu0"])
    close(bwd["dW_gu"][1], names["dW_gu1"])
    close(bwd["dW_d"][0], names["dW_d0"])
    close(bwd["dW_d"][1], names["dW_d1"])
    close(bwd["d_logits"][0], names["d_logits"])


def _grouped_blocks():
    blocks, cur = [], None
    for line in _lines("routing_grouped.txt"):
        key, _, rest = line.partition(" ")
        if key == "grouped":
            f = rest.split()
            cur = {"k": int(f[1]), "E": int(f[3]), "n_group": int(f[5]), "topk_group": int(f[7]),
                   "scale": float(f[9]), "logits": [], "idx": [], "w": []}
            blocks.append(cur)
        elif key == "bias":
            cur["bias"] = [float(t) for t in rest.split()]
        elif key == "token":
            lg, _, out = rest.partition("->")
            idx, _, w = out.partition("|")
            cur["logits"].append([_expr(t) for t in lg.split()])
            cur["idx"].append([int(t) for t in idx.split()])
            cur["w"].append([_expr(t) for t in w.split()])
        elif key == "split_sizes":
            cur["split"] = [int(t) for t in rest.split()]
    return blocks


@pytest.mark.parametrize("block", _grouped_blocks())
def test_grouped_routing_by_hand(block):
    logits = np.array(block["logits"], np.float32)
    idx, w = om.route_grouped(logits, block["k"], block["n_group"], block["topk_group"], np.array(block["bias"]),
                              block["scale"], np.float64)
    assert np.array_equal(idx, np.array(block["idx"]))
    np.testing.assert_allclose(w, np.array(block["w"]), rtol=0, atol=1e-6)   # fp32 logits
    split, _, _, _ = om.dispatch(idx, block["E"])
    assert list(split) == block["split"]
