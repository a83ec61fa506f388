"""Write sampled oracle outputs of the full-size workloads to tests/golden/full_<name>.npz.

Calls only the oracle (and the shared input generator). For each workload and each
sampled item the whole fp64 encoder runs on the CPU; the file keeps a fixed set of token
rows (first rows incl. any CLS, tile edges, the ragged last rows and a seeded random
spread) as float32, together with the item index and the row ids.

    python tests/golden/make_full_goldens.py [name ...]
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
from configs import WORKLOADS  # noqa: E402

SEED = 0
N_RANDOM_ROWS = 12


def sample_rows(N: int) -> np.ndarray:
    fixed = [0, 1, 2, 127, 128, 129, N // 2, N - 129, N - 128, N - 2, N - 1]
    rng = np.random.default_rng(1234 + N)
    rnd = rng.choice(N, size=N_RANDOM_ROWS, replace=False)
    return np.unique(np.clip(np.array(fixed + list(rnd)), 0, N - 1))


def main(names):
    for name in names:
        cfg, dtype, batches, (T, H, W) = WORKLOADS[name]
        B = max(batches)
        items = sorted({0, B - 1})
        N = oracle.n_tokens(cfg, T, H, W)
        rows = sample_rows(N)
        item_size = T * 3 * H * W
        outs = []
        for b in items:
            pix = np.empty((1, T, 3, H, W), dtype=np.float32)
            synth.lib().jsynth_api_pixels(SEED, b * item_size, item_size, pix.ctypes.data)
            t0 = time.time()
            y = oracle.encode(cfg, SEED, dtype == "bf16", pix)[0]
            print(f"{name} item {b}: N={N} oracle {time.time() - t0:.1f} s", flush=True)
            outs.append(y[rows].astype(np.float32))
        np.savez_compressed(os.path.join(HERE, f"full_{name}.npz"), rows=rows, items=np.array(items),
                            batch=B, seed=SEED, tokens=np.stack(outs))


if __name__ == "__main__":
    main(sys.argv[1:] or list(WORKLOADS))
