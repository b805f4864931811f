"""How far the mixed_fp8 recipe alone moves the Whisper large-v3 encoder (oracle only, CPU).

The showcase site's mixed_fp8 preset ("The Approach": encoder_attn_qkv and
encoder_ffn in E4M3, weights and activations, one absmax scale per tensor)
is applied inside the float64 oracle itself, with every other step exact, and
compared with the unquantised float64 oracle on the same seeded chunk and the
same random-init weights (the batch-32 workload's last chunk).  No GPU code is
involved: the gap measured here is the quantisation's own, so it is a floor
under the gap of ANY implementation of the recipe from the unquantised oracle.

It grows with depth and passes a relative L2 of 6e-2 within the first five of
the 32 layers, which is why the mixed_fp8 tolerance is applied per layer and
against the oracle of the same (quantised) pipeline."""
import numpy as np
import pytest

from oracle import encoder as oenc
from oracle import frontend as ofe
import synthetic

pytestmark = pytest.mark.slow


def test_quantisation_alone_exceeds_6e2_within_five_layers():
    dims = synthetic.LARGE_V3
    n = 5
    w = synthetic.encoder_weights(dims, synthetic.SEED_LARGE_B32, "bf16", n_layers=n)
    x0 = oenc.conv_stem(ofe.log_mel(synthetic.tone_chunk(synthetic.SEED_LARGE_B32 + 31), dims.n_mels), w)
    plain, quant = [], []
    oenc.encoder(x0, w, dims.n_heads, final_ln=False, capture=plain)
    oenc.encoder(x0, w, dims.n_heads, final_ln=False, capture=quant, fp8_sites=oenc.MIXED_FP8)
    gap = [float(np.linalg.norm(q - p) / np.linalg.norm(p)) for q, p in zip(quant, plain)]
    print("relative L2 of the E4M3 oracle from the unquantised oracle after each layer:",
          " ".join(f"{g:.3e}" for g in gap))
    assert all(b > a for a, b in zip(gap, gap[1:]))           # the gap accumulates layer by layer
    assert gap[0] > 3e-2                                      # one layer already takes half the budget
    assert gap[-1] > 6e-2                                     # five layers exceed it


def _drift():
    import json
    import os
    with open(os.path.join(os.path.dirname(__file__), "golden", "fp8_drift.json")) as fh:
        return json.load(fh)


def test_stored_drift_comes_from_this_oracle():
    # tests/golden/fp8_drift.json is written by tests/golden/make_fp8_drift.py (oracle only, ~25 min);
    # its first layer is recomputed here, so a change of the oracle's arithmetic shows up as a mismatch
    from oracle import fp8 as ofp8
    d = _drift()
    assert len(d["per_layer"]) == 32
    dims = synthetic.LARGE_V3
    w = synthetic.encoder_weights(dims, d["workload"]["weights_seed"], "bf16", n_layers=1)
    x0 = oenc.conv_stem(ofe.log_mel(synthetic.tone_chunk(d["workload"]["chunk_seed"]), dims.n_mels), w)
    L = w["layers"][0]
    plain = oenc.encoder_layer(x0, L, dims.n_heads)
    q = oenc.encoder_layer(x0, L, dims.n_heads, oenc.MIXED_FP8)
    qb = ofp8.round_bf16(q)
    rel = lambda a, b: float(np.linalg.norm(a - b) / np.linalg.norm(b))  # noqa: E731
    assert abs(rel(q, plain) - d["per_layer"][0]["e4m3_vs_plain"]) < 1e-12
    assert abs(rel(qb, q) - d["per_layer"][0]["e4m3_b_vs_e4m3"]) < 1e-12


def test_stored_drift_shape():
    # both gaps grow with depth; bf16 storage of the residual stream alone, amplified by the E4M3
    # decisions downstream of it, moves the E4M3 oracle by several 1e-2 over the 32 layers
    d = _drift()
    e, b = [r["e4m3_vs_plain"] for r in d["per_layer"]], [r["e4m3_b_vs_e4m3"] for r in d["per_layer"]]
    assert b[0] < 2e-3 < 1e-2 < b[1]                      # one bf16 rounding, then the first E4M3 layer after it
    assert max(b[-4:]) > 4e-2 and e[-1] > 6e-2
    assert d["final_ln"]["e4m3_vs_plain"] > 6e-2
