"""Write oracle outputs of the full-size V-JEPA 2 ViT-L SSv2 attentive-pool head to
tests/golden/full_head_vjepa2_vitl16_ssv2.npz.

Calls only the oracle and the shared input generator: 8 items of 2048 encoder tokens N(0, 1);
items 0 and 7 run through the whole fp64 head (3 pooler layers, cross attention, MLP,
174-way classifier); the file keeps their pooled features and logits as float32.

    python tests/golden/make_head_golden.py
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
from configs import HEAD_VJEPA2_L16_SSV2, HEAD_WORKLOAD  # noqa: E402

SEED = 5


def main():
    B, N, D = max(HEAD_WORKLOAD["batches"]), HEAD_WORKLOAD["tokens"], HEAD_VJEPA2_L16_SSV2.embed_dim
    tokens = synth.fill(SEED, "input.enc_tokens", synth.NORMAL, 0.0, 1.0, (B, N, D))
    items = [0, B - 1]
    pooled, logits = [], []
    for b in items:
        t0 = time.time()
        p, l = oracle.attentive_head(HEAD_VJEPA2_L16_SSV2, 0, True, tokens[b:b + 1])
        print(f"head item {b}: {time.time() - t0:.1f} s", flush=True)
        pooled.append(p[0].astype(np.float32))
        logits.append(l[0].astype(np.float32))
    np.savez_compressed(os.path.join(HERE, "full_head_vjepa2_vitl16_ssv2.npz"), batch=B, tokens=N, seed=SEED,
                        items=np.array(items), pooled=np.stack(pooled), logits=np.stack(logits))


if __name__ == "__main__":
    main()
