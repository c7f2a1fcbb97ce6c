"""Pins of the oracle's quantize-then-dispatch step (CPU only).

The routing (counts, offsets, both row maps) is checked against cases worked
out by hand in tests/golden/dispatch_routing.txt; an unstable order, a wrong
padding rule (an off-by-one at exactly 128 tokens, or padding an empty expert)
or a dropped token that still takes a row each fails one of them.  The codes
are pinned by relations to the already-pinned 1x128 quantizer: a routed row
holds exactly the quantization of its token's row, a padding row holds codes
0 and scale 1."""
import os

import numpy as np
import pytest
import torch

import oracle
import workloads as wl
from workloads import bf16_bits

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "dispatch_routing.txt")


def _items(tokens):
    out = []
    for it in tokens:
        if "*" in it:
            v, n = it.split("*")
            out.extend([-1 if v == "-" else int(v)] * int(n))
        elif ".." in it:
            a, b = it.split("..")
            out.extend(range(int(a), int(b) + 1))
        elif it == "-":
            out.append(-1)
        else:
            out.append(int(it))
    return out


def _cases():
    cases, cur = {}, None
    with open(GOLDEN) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if not line:
                continue
            key, *rest = line.split()
            if key == "case":
                cur = cases.setdefault(rest[0], {"row_token": []})
            elif key == "E":
                cur["E"] = int(rest[0])
            elif key == "row_token":
                r0, r1 = int(rest[0]), int(rest[1])
                vals = _items(rest[3:])
                assert rest[2] == ":" and len(vals) == r1 - r0 + 1, line
                cur["row_token"].append((r0, r1, vals))
            else:
                cur[key] = _items(rest)
    return cases


CASES = _cases()


def test_golden_cases_are_complete():
    assert set(CASES) == {"seven_tokens", "boundary_counts", "dropped_tokens"}
    for c in CASES.values():
        n = c["offsets"][-1]
        covered = sorted(r for r0, r1, _ in c["row_token"] for r in range(r0, r1 + 1))
        assert covered == list(range(n)), "row_token segments must cover every row once"


@pytest.mark.parametrize("name", sorted(CASES))
def test_dispatch_routing_matches_hand_worked_case(name):
    c = CASES[name]
    expert = np.array(c["expert"], np.int64)
    T, K = expert.size, 128
    x = np.random.default_rng(len(name)).standard_normal((T, K)).astype(np.float32)
    q, s, offsets, counts, token_row, row_token, dropped = oracle.dispatch(x, expert, c["E"])
    assert counts.tolist() == c["counts"]
    assert offsets.tolist() == c["offsets"]
    assert token_row.tolist() == c["token_row"]
    for r0, r1, vals in c["row_token"]:
        assert row_token[r0:r1 + 1].tolist() == vals, f"rows {r0}..{r1}"
    assert dropped == int(np.sum((expert < 0) | (expert >= c["E"])))


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_dispatched_rows_are_the_tokens_quantized(dtype):
    """Quantization is row-wise, so dispatching commutes with it: routed rows
    equal the 1x128 quantizer's rows of their tokens; padding rows are a
    quantized zero row (codes 0, scale 1)."""
    T, K, E = 700, 384, 9
    expert = np.random.default_rng(5).integers(0, E, T)
    expert[expert == 4] = 6                                 # one empty expert
    xt = wl.random_matrix((T, K), seed=6, dtype=dtype)
    x = bf16_bits(xt) if dtype == torch.bfloat16 else xt.numpy()
    q, s, offsets, counts, token_row, row_token, dropped = oracle.dispatch(x, expert, E)
    assert dropped == 0 and counts[4] == 0
    assert np.array_equal(counts, np.bincount(expert, minlength=E))
    assert np.all(np.diff(offsets) % 128 == 0)
    qx, sx = oracle.quant_act_1x128(x)
    routed = row_token >= 0
    assert np.array_equal(q[routed], qx[row_token[routed]])
    assert np.array_equal(s[:, routed], sx[:, row_token[routed]])
    assert np.all(q[~routed] == 0) and np.all(s[:, ~routed] == 1.0)
    assert np.array_equal(row_token[token_row], np.arange(T))   # the two maps are inverse
    for e in range(E):                                           # stable inside each expert
        rows = token_row[expert == e]
        assert np.all(np.diff(rows) == 1) and (rows.size == 0 or rows[0] == offsets[e])


def test_dispatch_empty_and_all_dropped():
    x = np.zeros((0, 128), np.float32)
    q, s, offsets, counts, token_row, row_token, dropped = oracle.dispatch(
        x, np.zeros(0, np.int64), 3)
    assert offsets.tolist() == [0, 0, 0, 0] and q.shape == (0, 128) and dropped == 0
    x = np.ones((4, 128), np.float32)
    q, s, offsets, counts, token_row, row_token, dropped = oracle.dispatch(
        x, np.array([3, 7, -2, 3]), 3)
    assert offsets.tolist() == [0, 0, 0, 0] and token_row.tolist() == [-1] * 4
    assert dropped == 4
