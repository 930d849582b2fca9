"""Write the regression fixture ``oracle_small.json`` from the float64 oracle.

Run from the repository root:  python tests/golden/make_golden.py

The fixture pins the oracle to its own committed behaviour, so that a later
change to its arithmetic shows up as a test failure (and has to be justified
by the passage it follows).  Inputs come from the shared seeded generator;
every expected value is computed by ``oracle`` alone.
"""
import json
import os
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(os.path.dirname(HERE))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

import oracle  # noqa: E402
from exact_attention_58_gb300.workloads import make_inputs  # noqa: E402

CASES = [
    # name, B, H, N, d, causal, key_len_range, p
    ("plain", 1, 2, 9, 4, False, None, 0.0),
    ("causal_pad_dropout", 2, 2, 11, 8, True, (5, 11), 0.25),
]


def main():
    out = {"generator": "exact_attention_58_gb300.workloads.make_inputs (bf16 inputs)",
           "cases": []}
    for idx, (name, B, H, N, d, causal, klr, p) in enumerate(CASES):
        inp = make_inputs(B, H, N, d, dtype=torch.bfloat16, gen_seed=777 + idx, causal=causal,
                          key_len_range=klr, dropout_p=p, dropout_seed_value=4242 + idx)
        q, k, v, do = (t.double().numpy() for t in (inp.q, inp.k, inp.v, inp.do))
        kl = None if inp.key_lens is None else inp.key_lens.numpy()
        O, LSE = oracle.attn_fwd(q, k, v, inp.scale, causal, kl, p, inp.seed)
        dQ, dK, dV, D = oracle.attn_bwd(q, k, v, do, inp.scale, causal, kl, p, inp.seed)
        out["cases"].append({
            "name": name, "B": B, "H": H, "N": N, "d": d, "causal": causal,
            "key_lens": None if kl is None else kl.tolist(), "dropout_p": p, "seed": inp.seed,
            "scale": inp.scale, "q": q.ravel().tolist(), "k": k.ravel().tolist(),
            "v": v.ravel().tolist(), "do": do.ravel().tolist(),
            "O": O.ravel().tolist(), "LSE": [x if np.isfinite(x) else None for x in LSE.ravel()],
            "dQ": dQ.ravel().tolist(), "dK": dK.ravel().tolist(), "dV": dV.ravel().tolist(),
        })
    with open(os.path.join(HERE, "oracle_small.json"), "w") as f:
        json.dump(out, f, indent=0)


if __name__ == "__main__":
    main()
