"""Writes fp8_drift.json: how far the mixed_fp8 recipe and bf16 storage move the float64 oracle.

Calls only oracle/ (and the seeded input generators).  The showcase site's mixed_fp8 preset ("The
Approach": encoder_attn_qkv and encoder_ffn in E4M3, one absmax scale per tensor) on the batch-32
workload's last chunk (seed 2031, weights seed 2000), large-v3, 32 layers:
  plain   the unquantised float64 oracle
  e4m3    the oracle with E4M3 operands at the qkv and ffn sites (the oracle of the mixed_fp8 pipeline)
  e4m3_b  the same, with the residual stream rounded to bf16 after every layer (the storage a bf16
          pipeline gives it), and otherwise identical arithmetic
Relative L2 after every layer and after the final LayerNorm.  Run:  python tests/golden/make_fp8_drift.py
(about 15 minutes on 8 cores)."""
import json
import os
import sys

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(os.path.dirname(HERE)))

import synthetic  # noqa: E402
from oracle import encoder as oenc  # noqa: E402
from oracle import fp8 as ofp8  # noqa: E402
from oracle import frontend as ofe  # noqa: E402


def rel(a, b):
    return float(np.linalg.norm(a - b) / np.linalg.norm(b))


def main():
    dims = synthetic.LARGE_V3
    seed, chunk = synthetic.SEED_LARGE_B32, synthetic.SEED_LARGE_B32 + 31
    w = synthetic.encoder_weights(dims, seed, "bf16")
    x0 = oenc.conv_stem(ofe.log_mel(synthetic.tone_chunk(chunk), dims.n_mels), w)
    plain, q, qb = x0.copy(), x0.copy(), x0.copy()
    rows = []
    for i, L in enumerate(w["layers"]):
        plain = oenc.encoder_layer(plain, L, dims.n_heads)
        q = oenc.encoder_layer(q, L, dims.n_heads, oenc.MIXED_FP8)
        qb = ofp8.round_bf16(oenc.encoder_layer(qb, L, dims.n_heads, oenc.MIXED_FP8))
        rows.append({"layer": i, "e4m3_vs_plain": rel(q, plain), "e4m3_b_vs_e4m3": rel(qb, q)})
        print(rows[-1], flush=True)
    ln = lambda h: oenc.layer_norm(h, w["ln_post_g"], w["ln_post_b"])  # noqa: E731
    final = {"e4m3_vs_plain": rel(ln(q), ln(plain)), "e4m3_b_vs_e4m3": rel(ln(qb), ln(q))}
    out = {"what": "relative L2 between float64 oracle chains, large-v3, 32 layers; see make_fp8_drift.py",
           "workload": {"weights_seed": seed, "chunk_seed": chunk}, "per_layer": rows, "final_ln": final}
    with open(os.path.join(HERE, "fp8_drift.json"), "w") as fh:
        json.dump(out, fh, indent=1)
    print(final)


if __name__ == "__main__":
    main()
