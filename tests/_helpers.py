"""Helpers shared by the GPU parity tests (comparison rules, device transfer, parity record)."""
import json
import os

import numpy as np

NEAR_TIE = 5e-2           # top-2 perturbed-logit gap below which a token may differ
LOGIT_TOL = 2e-2          # max abs error of base logits (bf16 inputs, fp32 accumulation)
# Bound on the share of compared positions that may diverge at a near tie.  The GPU works in
# fp32 and the oracle in fp64: their perturbed values differ by ~1e-5, so a token can flip only
# where the top-2 gap is that small, a fraction ~1e-5 of positions (the gap of a Gumbel-max has
# density ~1 near 0).  A kernel that mishandled near ties (a wrong tie order, a dropped noise
# term) would instead flip a good part of the ~5 % of positions whose gap is below 5e-2.
MAX_TIE_FRACTION = 0.01

# one entry per comparison: (kind, label, compared, near_tie); printed and written at session end
PARITY_RECORD = []


def to_dev(a, dev="cuda"):
    import torch
    if isinstance(a, np.ndarray):
        a = torch.from_numpy(np.ascontiguousarray(a))
    return a.to(dev)


def record_parity(kind, label, compared, near_tie):
    PARITY_RECORD.append((kind, label, int(compared), int(near_tie)))


def check_tie_share(compared, ties, what):
    allowed = max(1, int(MAX_TIE_FRACTION * compared))
    assert ties <= allowed, (f"{what}: {ties} near-tie divergences in {compared} compared positions "
                             f"(at most {allowed} allowed)")


def check_markov_parity(gpu_tokens, base_logits, anchor, w1, w2, temperature, seed, offset,
                        req_ids=None, label="", near_tie=NEAR_TIE, kind="markov"):
    """Teacher-forced comparison of a GPU token sequence with the oracle, every position.

    The oracle runs each step on the GPU's own previous token (its teacher-forced mode), so a
    near tie at one step does not change what the later steps condition on.  A position may
    differ only where the oracle's top-2 gap of perturbed values is below `near_tie`; such
    positions are counted, bounded by MAX_TIE_FRACTION of the compared positions, and recorded.
    Returns (compared, near_tie_divergences, oracle lse [Bs, N] on the GPU's prefix).
    """
    g = np.asarray(gpu_tokens).astype(np.int64)
    ref, gap, lse = oracle_markov_forced(base_logits, anchor, w1, w2, temperature, seed, offset, req_ids, g)
    compared, ties = compare_teacher_forced(g, ref, gap, near_tie)
    check_tie_share(compared, ties, label or kind)
    record_parity(kind, label, compared, ties)
    return compared, ties, lse


def oracle_markov_forced(base_logits, anchor, w1, w2, temperature, seed, offset, req_ids, forced):
    """The oracle's teacher-forced sampler over request chunks on a thread pool (numpy releases
    the interpreter lock in its array work); each chunk keeps its requests' counter ids."""
    import oracle
    from concurrent.futures import ThreadPoolExecutor
    L = np.asarray(base_logits)
    Bs = L.shape[0]
    req = np.arange(Bs) if req_ids is None else np.asarray(req_ids)
    anchor, temperature = np.asarray(anchor), np.asarray(temperature)
    step = 4
    chunks = [np.arange(c, min(Bs, c + step)) for c in range(0, Bs, step)]

    def run(ix):
        return oracle.markov_sample(L[ix], anchor[ix], w1, w2, temperature[ix], seed, offset,
                                    req_ids=req[ix], forced_tokens=forced[ix])

    with ThreadPoolExecutor(max(1, min(len(chunks), os.cpu_count() or 1))) as ex:
        parts = list(ex.map(run, chunks))
    return tuple(np.concatenate([p[k] for p in parts]) for k in range(3))


def compare_teacher_forced(gpu_tokens, ref_tokens, ref_gap, near_tie=NEAR_TIE):
    """Position-by-position comparison against teacher-forced oracle tokens.

    Returns (compared positions, near-tie divergences); raises on a mismatch at a gap of
    `near_tie` or more.
    """
    g = np.asarray(gpu_tokens)
    r = np.asarray(ref_tokens)
    diff = g != r
    bad = diff & (np.asarray(ref_gap) >= near_tie)
    if bad.any():
        b, i = (int(x[0]) for x in np.nonzero(bad))
        raise AssertionError(f"token mismatch at request {b} step {i}: gpu {g[b, i]} oracle {r[b, i]} "
                             f"(oracle top-2 gap {ref_gap[b, i]:.3g} >= {near_tie})")
    return int(g.size), int(diff.sum())


def parity_summary_lines():
    """Totals of the recorded comparisons per kind, one line each."""
    by = {}
    for kind, _, n, t in PARITY_RECORD:
        c = by.setdefault(kind, [0, 0, 0])
        c[0] += n
        c[1] += t
        c[2] += 1
    return [f"parity {k}: {c[2]} comparisons, {c[0]} positions compared, {c[1]} near-tie divergences"
            for k, c in sorted(by.items())]


def write_parity_record(path):
    os.makedirs(os.path.dirname(os.path.abspath(path)), exist_ok=True)
    with open(path, "w") as f:
        json.dump({"entries": [{"kind": k, "test": lbl, "compared": n, "near_tie": t}
                               for k, lbl, n, t in PARITY_RECORD],
                   "max_tie_fraction": MAX_TIE_FRACTION}, f, indent=1)
