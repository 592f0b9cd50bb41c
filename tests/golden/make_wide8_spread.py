"""Write wide8_accumulation_spread.json: how far the oracle's own layer-streamed
bf16-operand step moves between fp32 and fp64 accumulation on the wide-8
parity inputs (8 layers, d_model 16384; parameters from seed 3, the two
sequences of seeds 3 and 4).

Both evaluations round every matrix-product operand to bf16 and nothing else;
they differ only in the precision of the sums. Their distance is the part of
the loss, the logits and the gradients of the first and last blocks, wte, wpe
and ln_f that fp32 accumulation leaves undetermined. Calls only the oracle and
the seeded input generator; needs ~170 GB of host memory and tens of
CPU-minutes.

    python tests/golden/make_wide8_spread.py
"""
import json
import os
import sys

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
sys.path.insert(0, ROOT)

from oracle import gpt2 as O  # noqa: E402
from tile_task_transformer_gb300 import synth  # noqa: E402

L, D, H, F, V, S, SEED = 8, 16384, 128, 65536, 50257, 1024, 3


def main():
    names = synth.param_names_shapes(L, D, F, V, S)
    index = {n: (i, sh) for i, (n, sh) in enumerate(names)}

    def gen(n):
        i, sh = index[n]
        return synth.gpt2_tensor(SEED, i, n, sh)

    head = {n: gen(n) for n in ("wte", "wpe", "ln_f.g", "ln_f.b")}
    layers = []
    for l in range(L):
        t = {}
        for k in ("ln1.g", "ln1.b", "qkv.w", "qkv.b", "o.w", "o.b", "ln2.g", "ln2.b", "fc.w", "fc.b",
                  "proj.w", "proj.b"):
            a = gen(f"h{l}.{k}")
            t[k] = O.bf16_bits(a) if k.endswith(".w") else a
        layers.append(t)

    def layer_params(l):
        return {k: (O.from_bf16_bits(v) if k.endswith(".w") else v) for k, v in layers[l].items()}

    seqs = np.concatenate([synth.token_windows(SEED, 1, S, V), synth.token_windows(SEED + 1, 1, S, V)])
    two = O.GPT2Config(n_layer=L, d_model=D, n_head=H, d_ff=F, vocab=V, seq=S, batch=2)
    runs = {}
    for dt in (np.float64, np.float32):
        loss, cache = O.forward_bf16_streamed(two, layer_params, head, seqs, dtype=dt)
        z = cache["z"].astype(np.float32)
        g = O.backward_bf16_streamed(two, layer_params, head, cache, want={0, L - 1}, dtype=dt,
                                     grad_dtype=np.float32)
        del cache
        runs[dt] = (float(loss), z, g)
    l64, z64, g64 = runs[np.float64]
    l32, z32, g32 = runs[np.float32]
    zd, zr = z32.astype(np.float64), z64.astype(np.float64)
    out = {"what": "layer-streamed bf16-operand oracle step, fp32 vs fp64 accumulation, wide-8 parity "
                   "inputs (params seed 3, sequences seeds 3 and 4)",
           "loss_fp32": l32, "loss_fp64": l64,
           "logits": {"two_norm": float(np.linalg.norm(zd - zr) / np.linalg.norm(zr)),
                      "max_norm": float(np.abs(zd - zr).max() / np.abs(zr).max())},
           "tensors": {}}
    for n in g64:
        a, r = g32[n].astype(np.float64), g64[n].astype(np.float64)
        out["tensors"][n] = {"two_norm": float(np.linalg.norm(a - r) / np.linalg.norm(r)),
                             "max_norm": float(np.abs(a - r).max() / np.abs(r).max())}
    path = os.path.join(os.path.dirname(os.path.abspath(__file__)), "wide8_accumulation_spread.json")
    with open(path, "w") as fh:
        json.dump(out, fh, indent=1, sort_keys=True)
    print(path)


if __name__ == "__main__":
    main()
