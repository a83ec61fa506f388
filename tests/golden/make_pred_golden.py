"""Write sampled oracle outputs of the full-size V-JEPA 2 ViT-L masked predictor to
tests/golden/full_pred_vjepa2_vitl16.npz.

Calls only the oracle and the shared input generator. The workload: the 8 x 16 x 16 position
grid of a 16 x 256^2 clip (2048 tokens), 8 items of encoder tokens N(0, 1) from the generator;
even items take the pages' split (context = the first 1024 tokens, targets = the last 1024), odd
items a seeded random half / half split. Items 0 and 7 run through the whole fp64 predictor; the
file keeps a fixed set of target rows of each (tile edges, the ragged end, a seeded spread) as
float32, with all the ids.

    python tests/golden/make_pred_golden.py
"""
import os
import sys
import time

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(os.path.dirname(HERE)))
sys.path.insert(0, os.path.dirname(HERE))

import oracle  # noqa: E402
import synth  # noqa: E402
from configs import PRED_VJEPA2_L16, PRED_WORKLOAD  # noqa: E402

SEED = 3


def masks(B, n_pos, n_ctx, n_tgt):
    ctx, tgt = [], []
    rng = np.random.default_rng(2024)
    for b in range(B):
        order = np.arange(n_pos) if b % 2 == 0 else rng.permutation(n_pos)
        ctx.append(order[:n_ctx])
        tgt.append(order[n_ctx:n_ctx + n_tgt])
    return np.array(ctx, dtype=np.int32), np.array(tgt, dtype=np.int32)


def main():
    grid = PRED_WORKLOAD["grid"]
    B = max(PRED_WORKLOAD["batches"])
    n_pos = int(np.prod(grid))
    ctx, tgt = masks(B, n_pos, PRED_WORKLOAD["n_ctx"], PRED_WORKLOAD["n_tgt"])
    enc = synth.fill(SEED, "input.enc_tokens", synth.NORMAL, 0.0, 1.0, (B, n_pos, PRED_VJEPA2_L16.enc_dim))
    n_tgt = tgt.shape[1]
    rng = np.random.default_rng(99)
    rows = np.unique(np.concatenate([[0, 1, 127, 128, 129, n_tgt // 2, n_tgt - 2, n_tgt - 1],
                                     rng.choice(n_tgt, 12, replace=False)]))
    items = [0, B - 1]
    outs = []
    for b in items:
        t0 = time.time()
        y = oracle.predict(PRED_VJEPA2_L16, 0, True, enc[b:b + 1], ctx[b:b + 1], tgt[b:b + 1], grid[1:])[0]
        print(f"predictor item {b}: {time.time() - t0:.1f} s", flush=True)
        outs.append(y[rows].astype(np.float32))
    np.savez_compressed(os.path.join(HERE, "full_pred_vjepa2_vitl16.npz"), grid=np.array(grid), batch=B, seed=SEED,
                        ctx=ctx, tgt=tgt, rows=rows, items=np.array(items), out=np.stack(outs))


if __name__ == "__main__":
    main()
