"""Pins of the greedy-verification oracle: hand-worked cases, brute force over every draft of
a tiny vocabulary, the target's own greedy continuation, and invalid inputs."""
import itertools

import numpy as np

from oracle import verify_greedy, row_argmax


def _read_cases(path):
    cases, cur = [], None
    for line in open(path):
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        key, _, val = line.partition(" ")
        if key == "case":
            cur = {"name": val}
            cases.append(cur)
        elif key == "rows":
            cur["rows"] = np.array([[float(t) for t in r.split(",")] for r in val.split("|")])
        elif key == "draft":
            cur["draft"] = np.array([int(t) for t in val.split()])
        elif key == "length":
            cur["length"] = None if val == "-" else int(val)
        elif key == "expect":
            n, toks = val.split("|")
            cur["nacc"] = int(n)
            cur["out"] = np.array([int(t) for t in toks.split()])
    return cases


def test_hand_worked_cases(golden_dir):
    cases = _read_cases(golden_dir / "greedy_worked.txt")
    assert len(cases) == 9
    for c in cases:
        lengths = None if c["length"] is None else np.array([c["length"]])
        out, nacc = verify_greedy(c["rows"][None], c["draft"][None], lengths)
        assert nacc[0] == c["nacc"], c["name"]
        np.testing.assert_array_equal(out[0], c["out"], err_msg=c["name"])


def test_brute_force_over_all_drafts_of_a_tiny_vocabulary():
    """For every draft block the accepted prefix is exactly the longest prefix matching the
    per-row argmaxes, and the appended token is the argmax of the next row."""
    rng = np.random.default_rng(3)
    V, gamma = 3, 3
    for _ in range(20):
        rows = rng.integers(0, 4, size=(gamma + 1, V)).astype(np.float64)   # many ties
        am = [int(np.flatnonzero(r == r.max())[0]) for r in rows]
        for draft in itertools.product(range(V), repeat=gamma):
            out, nacc = verify_greedy(rows[None], np.array(draft)[None])
            k = 0
            while k < gamma and draft[k] == am[k]:
                k += 1
            assert nacc[0] == k
            assert list(out[0, :k]) == list(draft[:k]) and out[0, k] == am[k]
            assert np.all(out[0, k + 1:] == -1)


def test_output_is_the_targets_greedy_continuation():
    """Drafting the target's own argmaxes accepts everything and appends the bonus argmax."""
    rng = np.random.default_rng(4)
    t = rng.standard_normal((5, 7, 50))
    x = np.argmax(t[:, :6], axis=2)
    out, nacc = verify_greedy(t, x)
    assert np.all(nacc == 6)
    np.testing.assert_array_equal(out[:, 6], np.argmax(t[:, 6], axis=1))


def test_invalid_tokens_and_lengths_give_minus_one():
    t = np.ones((3, 3, 4))
    out, nacc = verify_greedy(t, np.array([[0, 5], [0, 0], [-1, 0]]), np.array([2, 3, 1]))
    assert np.all(out == -1) and np.all(nacc == 0)


def test_row_argmax_rules():
    assert row_argmax(np.array([1.0, 3.0, 3.0])) == 1
    assert row_argmax(np.array([np.nan, 0.5, np.nan])) == 1
    assert row_argmax(np.array([np.nan, np.nan])) == 0
    assert row_argmax(np.array([-np.inf, -np.inf])) == 0
