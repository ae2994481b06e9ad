"""Writes closed_form_cases.json: small inputs whose loss, lse and gradients follow by hand.

Each case below is its derivation written out with ``math.log`` and plain arithmetic (no
oracle, no NumPy, no loops over a vocabulary beyond filling in the constant entries), so a
reader can check every stored value against the formulas of the loss:

    lse_t = log sum_v exp(s_tv / tau),  p_t = softmax(z_t / tau) over the K slots,
    KL_t = sum_k p_tk (log p_tk - (s_{t,id_tk} / tau - lse_t)),  L = tau^2 sum_t w_t KL_t,
    dS_tv = tau w_t (q_tv - ptilde_tv),  dH = dS W,  dW = dS^T H,

with w_t = 1/N over the valid tokens (or 1/(S N_s) for the sequence mean; N replaced by the
whole batch's count when the case gives one).

    python tests/golden/make_closed_form_cases.py          # prints the differences, if any
    python tests/golden/make_closed_form_cases.py --write  # rewrites the JSON file
"""
from __future__ import annotations

import json
import math
import os
import sys

PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "closed_form_cases.json")
SOURCE = ("Closed-form special cases of the loss defined in 'Efficient Knowledge Distillation for LLMs: "
          "Offline Top-K Logits and a Fused Chunked KL Loss' (section 'Two systems changes', dense KL "
          "baseline), derived by hand; the pages print no worked example. Values are the derivations "
          "evaluated in float64 by tests/golden/make_closed_form_cases.py.")

LN2, LN3, LN5, LN8 = math.log(2.0), math.log(3.0), math.log(5.0), math.log(8.0)


def outer(col, row):
    return [[a * b for b in row] for a in col]


def uniform_row_dS(scale, ids_p, V=8):
    """scale * (1/V - ptilde) for a uniform student (W = 0) over V ids."""
    ds = [scale * (1.0 / V)] * V
    for v, p in ids_p:
        ds[v] = scale * (1.0 / V - p)
    return ds


def uniform_student():
    kl = LN8 + 0.75 * math.log(0.75) + 0.25 * math.log(0.25)
    H = [0.5, -1.0]
    dS = uniform_row_dS(1.0, [(5, 0.75), (2, 0.25)])
    return dict(
        name="uniform_student",
        derivation="W = 0 gives s = 0, so q = 1/V and lse = ln V for any tau. z = [ln 3, 0], tau = 1 gives "
                   "p = [3/4, 1/4]. KL = sum_k p_k ln p_k + ln V. dS = tau/N (q - ptilde) = 1/8 - ptilde; "
                   "dH = dS W = 0; dW = dS^T H.",
        T=1, d=2, V=8, K=2, tau=1.0, H=[H], W=[[0.0, 0.0]] * 8, ids=[[5, 2]], z=[[LN3, 0.0]], mask=[1],
        loss=kl, lse=[LN8], dH=[[0.0, 0.0]], dW=outer(dS, H))


def tempered_two_slot():
    tau = 2.0
    kl = (2.0 / 3.0) * math.log(4.0 / 3.0) + (1.0 / 3.0) * LN2
    dS = [2.0 * (1 / 6 - 1 / 3), 2.0 * (1 / 6), 2.0 * (1 / 6), 2.0 * (1 / 2 - 2 / 3)]
    return dict(
        name="tempered_two_slot",
        derivation="tau = 2, s = [0, 0, 0, 2 ln 3] so a = s/tau = [0, 0, 0, ln 3], exp(a) = [1, 1, 1, 3], "
                   "lse = ln 6, q = [1/6, 1/6, 1/6, 1/2]. ids = [3, 0], z = [2 ln 2, 0] so p = [2/3, 1/3]. "
                   "KL = 2/3 ln((2/3)/(1/2)) + 1/3 ln((1/3)/(1/6)) = 2/3 ln(4/3) + 1/3 ln 2; L = tau^2 KL. "
                   "dS = tau/N (q - ptilde) = 2 ([1/6,1/6,1/6,1/2] - [1/3,0,0,2/3]) = [-1/3, 1/3, 1/3, -1/3]; "
                   "dH = dS W = -(2/3) ln 3; dW = dS^T H.",
        T=1, d=1, V=4, K=2, tau=tau, H=[[1.0]], W=[[0.0], [0.0], [0.0], [2.0 * LN3]], ids=[[3, 0]],
        z=[[2.0 * LN2, 0.0]], mask=[1], loss=tau * tau * kl, lse=[math.log(6.0)], dH=[[-(2.0 / 3.0) * LN3]],
        dW=[[x] for x in dS])


def masked_second_row():
    u = uniform_student()
    return dict(
        name="masked_second_row",
        derivation="Row 0 is the uniform_student case; row 1 is masked, so N = 1, the loss and dW equal the "
                   "uniform_student values, dH of row 1 is 0 and lse of row 1 is still ln V = ln 8.",
        T=2, d=2, V=8, K=2, tau=1.0, H=[[0.5, -1.0], [3.0, 7.0]], W=[[0.0, 0.0]] * 8, ids=[[5, 2], [0, 1]],
        z=[[LN3, 0.0], [1.0, 2.0]], mask=[1, 0], loss=u["loss"], lse=[LN8, LN8], dH=[[0.0, 0.0], [0.0, 0.0]],
        dW=u["dW"])


def single_slot_cross_entropy():
    dS = [1.0 / 8.0, 2.0 / 8.0 - 1.0, 5.0 / 8.0]
    return dict(
        name="single_slot_cross_entropy",
        derivation="K = 1 gives p = 1, so KL = -ln q_id (cross-entropy). s = [0, ln 2, ln 5], exp(s) = [1, 2, 5], "
                   "lse = ln 8, id = 1: KL = -ln(2/8) = ln 4. dS = q - onehot = [1/8, -3/4, 5/8]; "
                   "dH = dS W = -(3/4) ln 2 + (5/8) ln 5; dW = dS^T H.",
        T=1, d=1, V=3, K=1, tau=1.0, H=[[1.0]], W=[[0.0], [LN2], [LN5]], ids=[[1]], z=[[0.25]], mask=[1],
        loss=math.log(4.0), lse=[LN8], dH=[[-0.75 * LN2 + 0.625 * LN5]], dW=[[x] for x in dS])


def two_packed_sequences_sequence_mean():
    kl0 = LN8 + 0.75 * math.log(0.75) + 0.25 * math.log(0.25)
    kl12 = LN8 + math.log(0.5)
    H = [[0.5, -1.0], [2.0, 1.0], [-1.0, 3.0]]
    dS = [uniform_row_dS(0.5, [(5, 0.75), (2, 0.25)]),
          uniform_row_dS(0.25, [(0, 0.5), (1, 0.5)]),
          uniform_row_dS(0.25, [(0, 0.5), (1, 0.5)])]
    dW = [[sum(dS[t][v] * H[t][j] for t in range(3)) for j in range(2)] for v in range(8)]
    return dict(
        name="two_packed_sequences_sequence_mean",
        derivation="Uniform student (W = 0, V = 8): q = 1/8, lse = ln 8. Token 0 (sequence 0) has p = [3/4, 1/4] "
                   "at ids [5, 2], KL_0 = ln 8 + 3/4 ln(3/4) + 1/4 ln(1/4); tokens 1 and 2 (sequence 1) have "
                   "p = [1/2, 1/2] at ids [0, 1], KL = ln 8 + ln(1/2) = ln 4. Sequence mean: "
                   "L = (KL_0 + (ln 4 + ln 4)/2) / 2, token weights w = [1/2, 1/4, 1/4]. "
                   "dS_t = tau w_t (q - ptilde_t); dH = dS W = 0; dW = dS^T H.",
        T=3, d=2, V=8, K=2, tau=1.0, H=H, W=[[0.0, 0.0]] * 8, ids=[[5, 2], [0, 1], [0, 1]],
        z=[[LN3, 0.0], [0.0, 0.0], [0.0, 0.0]], mask=[1, 1, 1], norm="sequences", seq_ids=[0, 1, 1],
        loss=(kl0 + (kl12 + kl12) / 2.0) / 2.0, lse=[LN8] * 3, dH=[[0.0, 0.0]] * 3, dW=dW)


def shard_with_batch_count():
    kl = LN8 + 0.75 * math.log(0.75) + 0.25 * math.log(0.25)
    H = [0.5, -1.0]
    dS = uniform_row_dS(0.25, [(5, 0.75), (2, 0.25)])
    return dict(
        name="shard_with_batch_count",
        derivation="The uniform_student row as one shard of a batch with 4 valid tokens (count = 4): the "
                   "shard's loss is KL / 4 with KL = ln 8 + 3/4 ln(3/4) + 1/4 ln(1/4), its token weight 1/4, "
                   "dS = 1/4 (1/8 - ptilde), dH = 0, dW = dS^T H: a quarter of uniform_student's.",
        T=1, d=2, V=8, K=2, tau=1.0, H=[H], W=[[0.0, 0.0]] * 8, ids=[[5, 2]], z=[[LN3, 0.0]], mask=[1], count=4,
        loss=kl / 4.0, lse=[LN8], dH=[[0.0, 0.0]], dW=outer(dS, H))


CASES = [uniform_student, tempered_two_slot, masked_second_row, single_slot_cross_entropy,
         two_packed_sequences_sequence_mean, shard_with_batch_count]


def cases():
    return {"source": SOURCE, "cases": [f() for f in CASES]}


def _diff(a, b, path="", tol=1e-14):
    if isinstance(a, dict) and isinstance(b, dict):
        out = [f"{path}: keys {sorted(set(a) ^ set(b))}"] if set(a) != set(b) else []
        for k in set(a) & set(b):
            out += _diff(a[k], b[k], f"{path}.{k}", tol)
        return out
    if isinstance(a, list) and isinstance(b, list):
        if len(a) != len(b):
            return [f"{path}: lengths {len(a)} != {len(b)}"]
        return [m for i, (x, y) in enumerate(zip(a, b)) for m in _diff(x, y, f"{path}[{i}]", tol)]
    if isinstance(a, float) or isinstance(b, float):
        return [] if abs(a - b) <= tol * max(1.0, abs(a), abs(b)) else [f"{path}: {a!r} != {b!r}"]
    return [] if a == b else [f"{path}: {a!r} != {b!r}"]


def differences(tol=1e-14):
    """Entries where the stored JSON and the derivations above disagree."""
    with open(PATH) as f:
        stored = json.load(f)
    return _diff(cases(), stored, "", tol)


if __name__ == "__main__":
    if "--write" in sys.argv:
        with open(PATH, "w") as f:
            json.dump(cases(), f, indent=1)
            f.write("\n")
    else:
        d = differences()
        print("\n".join(d) if d else "closed_form_cases.json matches its derivations")
