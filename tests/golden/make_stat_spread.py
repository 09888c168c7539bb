"""Writes stat_spread.json: how far fp32 tensor-core arithmetic by itself
moves the chained backward statistics s and s' (the relocated RMSNorm
statistics of "Reading notes on CODA", s3, "Eliminating the RMSNorm backward
kernel") away from their fp64 values. It calls only the oracle: the
storage-rounded rewritten forms run once in fp64 and once in the oracle's
fp32 mode (GEMMs through the tensor-core model tc_matmul, elementwise maps
in fp32), on the inputs and rows that the full-size GPU tests use, and the
max relative difference (||fp32 - fp64||_inf / ||fp64||_inf) is stored.
The GPU tests bound a chained statistic against the storage-rounded oracle by
max(1e-3, 2 x this spread).

Rows: the Llama-3-8B-shaped block on the rows its full-size test samples
(the first and last 32-row blocks and 16 scattered rows of M = 16384); the
Llama-3-1B-shaped block backward on its first 1024 rows (the GPU test checks
all 8192; the spread over 1024 rows was 1.3x that over 256).

Run:  python tests/golden/make_stat_spread.py   (about 40 s)
"""
import json
import os
import sys

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

from coda_inputs import WORKLOADS, block8b_inputs, mlp_block_inputs, positions  # noqa: E402
from oracle import coda_oracle as O  # noqa: E402
from tests._util import rows_8b_full  # noqa: E402

OUT = os.path.join(os.path.dirname(os.path.abspath(__file__)), "stat_spread.json")
ROWS_1B = 1024


def _maxrel(a, b):
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    return float(np.max(np.abs(a - b)) / np.max(np.abs(b)))


def spread_8b():
    sh = WORKLOADS["llama8b_block"]
    inp = block8b_inputs(sh)
    rows = rows_8b_full(sh.M)
    n = {k: O.to64(v[rows]) if v.dim() == 2 and v.shape[0] == sh.M else O.to64(v)
         for k, v in inp.items()}
    pos = positions(sh.M, sh.seq_len).numpy()[rows]
    res = {}
    for fp32 in (False, True):
        fr = O.block8b_fwd_reparam(n["o"], n["z"], n["Wo"], n["W1"], n["W2"], n["gamma2"],
                                   n["gamma1"], n["Wqkv"], pos, sh.n_rope_cols, sh.head_dim,
                                   sh.theta, store_bf16=True, fp32=fp32)
        res[fp32] = O.block8b_bwd_reparam(fr, n["o"], n["Wo"], n["W1"], n["W2"], n["gamma2"],
                                          n["gamma1"], n["Wqkv"], n["dqkv"], n["dres"], pos,
                                          sh.n_rope_cols, sh.head_dim, sh.theta, store_bf16=True,
                                          stat_only=True, fp32=fp32)
    return {"rows": f"{len(rows)} rows: 0..31, {sh.M - 32}..{sh.M - 1} and 16 sampled",
            "s1": _maxrel(res[True]["s1"], res[False]["s1"]),
            "s": _maxrel(res[True]["s"], res[False]["s"])}


def spread_1b():
    sh = WORKLOADS["llama1b_mlp_bwd"]
    inp = mlp_block_inputs(sh)
    n = {k: O.to64(v[:ROWS_1B]) if k in ("x", "z", "dout") else O.to64(v) for k, v in inp.items()}
    res = {}
    for fp32 in (False, True):
        f = O.mlp_fwd_reparam(n["x"], n["z"], n["W0"], n["W1"], n["W2"], n["gamma"],
                              store_bf16=True, fp32=fp32)
        res[fp32] = O.mlp_bwd_reparam(f, n["x"], n["W0"], n["W1"], n["W2"], n["gamma"], n["dout"],
                                      store_bf16=True, stat_only=True, fp32=fp32)
    return {"rows": f"0..{ROWS_1B - 1}", "s": _maxrel(res[True]["s"], res[False]["s"])}


def compute():
    return {"what": "max relative difference of the chained statistics between the oracle's "
                    "storage-rounded rewritten forms in fp32 (tensor-core model) and in fp64",
            "llama8b_block": spread_8b(), "llama1b_mlp_bwd": spread_1b()}


def main():
    out = compute()
    with open(OUT, "w") as f:
        json.dump(out, f, indent=1)
        f.write("\n")
    print(json.dumps(out, indent=1))


if __name__ == "__main__":
    main()
