"""Write wide4_accumulation_spread.json: how far the oracle's own bf16-operand
step moves between fp32 and fp64 accumulation on the wide-4 parity inputs.

Both evaluations round every matrix-product operand to bf16 and nothing else;
they differ only in the precision (and so the order effects) of the sums.
Their distance, per parameter tensor, is the part of a gradient that fp32
accumulation does not determine. Calls only the oracle and the seeded input
generator; needs ~80 GB of host memory and several CPU-minutes.

    python tests/golden/make_wide4_spread.py
"""
import json
import os
import sys

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
sys.path.insert(0, ROOT)

from oracle import gpt2 as O  # noqa: E402
from tile_task_transformer_gb300 import synth  # noqa: E402


def main():
    two = O.GPT2Config(n_layer=4, d_model=8192, n_head=64, d_ff=32768, vocab=50257, seq=1024, batch=2)
    params = synth.gpt2_params(3, two.n_layer, two.d_model, two.d_ff, two.vocab, two.seq)
    seqs = np.concatenate([synth.token_windows(3, 1, two.seq, two.vocab),
                           synth.token_windows(4, 1, two.seq, two.vocab)])
    l32, c = O.forward(two, params, seqs, dtype=np.float32, gemm_operands="bf16")
    g32 = O.backward_bf16_operands(two, params, c, dtype=np.float32)
    del c
    l64, c = O.forward(two, params, seqs, dtype=np.float64, gemm_operands="bf16")
    g64 = O.backward_bf16_operands(two, params, c, dtype=np.float64)
    del c
    out = {"what": "bf16-operand oracle step, fp32 vs fp64 accumulation, wide-4 parity inputs "
                   "(params seed 3, sequences seeds 3 and 4)",
           "loss_fp32": float(l32), "loss_fp64": float(l64), "tensors": {}}
    for n in g64:
        a, r = g32[n].astype(np.float64), g64[n]
        out["tensors"][n] = {
            "two_norm": float(np.linalg.norm(a - r) / np.linalg.norm(r)),
            "max_norm": float(np.abs(a - r).max() / np.abs(r).max()),
        }
    path = os.path.join(os.path.dirname(os.path.abspath(__file__)), "wide4_accumulation_spread.json")
    with open(path, "w") as fh:
        json.dump(out, fh, indent=1, sort_keys=True)
    print(path)


if __name__ == "__main__":
    main()
