"""The premise of the GPU test that rewrites positions with a residual add.

That test turns int64 positions `old` into `new` by adding bf16 words to the
positions buffer viewed as bf16.  Here, for every pair of positions in
[0, 256), the oracle's residual add and torch's eager bf16 add both give the
new position's bytes exactly.
"""
import numpy as np
import torch

import oracle
from helpers import position_delta_bf16, storage


def _all_pairs():
    old, new = np.meshgrid(np.arange(256, dtype=np.int64), np.arange(256, dtype=np.int64))
    return old.ravel(), new.ravel()


def test_position_delta_with_the_oracle_residual_add():
    old, new = _all_pairs()
    x = storage(position_delta_bf16(old, new)).reshape(len(old), 4)
    res = old.astype("<i8").view(np.uint16).reshape(len(old), 4)
    _, got, _ = oracle.add_rmsnorm(x, res, None, oracle.BF16, 1e-6)
    assert np.array_equal(np.ascontiguousarray(got).view("<i8").ravel(), new)


def test_position_delta_with_an_eager_bf16_add():
    old, new = _all_pairs()
    delta = position_delta_bf16(old, new).view(-1)
    pos = torch.from_numpy(old.copy()).view(torch.bfloat16)
    assert torch.equal((pos + delta).view(torch.int64), torch.from_numpy(new))
