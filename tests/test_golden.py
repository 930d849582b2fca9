"""The oracle against its committed regression anchor, and the IO model fixture."""
import json
import os

import numpy as np

import oracle

HERE = os.path.dirname(os.path.abspath(__file__))


def test_oracle_matches_committed_anchor():
    fx = json.load(open(os.path.join(HERE, "golden", "oracle_small.json")))
    for c in fx["cases"]:
        shp = (c["B"], c["H"], c["N"], c["d"])
        q, k, v, do = (np.array(c[n]).reshape(shp) for n in ("q", "k", "v", "do"))
        O, LSE = oracle.attn_fwd(q, k, v, c["scale"], c["causal"], c["key_lens"],
                                 c["dropout_p"], c["seed"])
        dQ, dK, dV, _ = oracle.attn_bwd(q, k, v, do, c["scale"], c["causal"], c["key_lens"],
                                        c["dropout_p"], c["seed"])
        np.testing.assert_allclose(O.ravel(), c["O"], rtol=0, atol=1e-12)
        ref_lse = np.array([-np.inf if x is None else x for x in c["LSE"]])
        np.testing.assert_allclose(LSE.ravel(), ref_lse, rtol=0, atol=1e-12)
        for got, name in ((dQ, "dQ"), (dK, "dK"), (dV, "dV")):
            np.testing.assert_allclose(got.ravel(), c[name], rtol=0, atol=1e-12)


def test_io_model_fixture_consistent():
    """The fused-attention IO formula the page prints, adapted to one LSE per
    row, equals the compulsory traffic the benchmark counts per head."""
    fx = json.load(open(os.path.join(HERE, "golden", "io_model.json")))
    from exact_attention_58_gb300.workloads import WORKLOADS
    import pytest
    bench = pytest.importorskip("bench")
    for w in WORKLOADS:
        N, d = w.N, w.d
        page = eval(fx["fused_attention"]["page_total"], {"N": N, "d": d})
        ours = eval(fx["fused_attention"]["this_library"].split(" (")[0], {"N": N, "d": d})
        assert ours == page - N
        es = 2 if w.dtype == "bf16" else 4
        assert bench.fwd_compulsory_bytes(w) == w.B * w.H * (4 * N * d * es + N * 4)
