"""GPU parity on random lists: 20 seeded cases, each a random storage mode,
a random mix of tensor sizes (empty, single-element, sub-vector, ragged and
multi-million), a random layout (16-byte aligned or skewed bases), with or
without clipping; half of the first 16 long enough for the interleaved
partition, the last 4 long enough (more than 8 rounds of tiles) for its
last rounds to be claimed at run time.  Every element of every buffer after
3 steps must match the oracle bit for bit."""
import numpy as np
import pytest

import parity_harness as H
from adamw_optimizer_step_sm_gb300 import workloads as W
from test_gpu_parity import _assert, _small

pytestmark = pytest.mark.gpu

MODES = [W.MODE_BF16_KAHAN, W.MODE_MIXED, W.MODE_REMAINDER, W.MODE_BF16_PLAIN,
         W.MODE_BF16_KAHAN_V32] + list(W.ANYPREC_MODES)


def _case(seed: int):
    rng = np.random.default_rng(1000 + seed)
    mode = int(rng.choice(MODES))
    n_t = int(rng.integers(3, 40))
    kinds = rng.integers(0, 4, n_t)
    sizes = []
    for k in kinds:
        if k == 0:
            sizes.append(int(rng.integers(0, 10)))
        elif k == 1:
            sizes.append(int(rng.integers(10, 5000)))
        elif k == 2:
            sizes.append(int(rng.integers(5000, 300_000)))
        else:
            sizes.append(int(rng.integers(300_000, 1_500_000)))
    if seed % 2:   # long: the interleaved partition
        sizes.append(int(rng.integers(6_000_000, 9_000_000)))
    clip = float(rng.choice([0.0, 0.3, 1.0]))
    layout = (8, 0) if rng.random() < 0.5 else (1, int(rng.integers(1, 8)))
    if seed >= 16:   # claimed last rounds
        sizes.insert(int(rng.integers(0, len(sizes) + 1)), int(rng.integers(30_000_000, 40_000_000)))
    return mode, sizes, clip, layout


@pytest.mark.parametrize("seed", range(20))
def test_random_list(seed):
    mode, sizes, clip, layout = _case(seed)
    w = _small(f"random{seed}", mode=mode, sizes=sizes, max_grad_norm=clip, steps=3)
    rep, log = H.run_parity(w, align_elems=layout[0], skew=layout[1])
    _assert(rep, log)
    assert rep.exact == rep.n, (mode, clip, layout)
