"""moe_permute_noalloc against moe_permute.

Some callers may not allocate device memory at all: a serving loop that gave
all of it to its own pool at start-up, or a plug-in host that only hands a
library its input and output buffers.  moe_permute_noalloc serves them with
a fixed static scratch array instead of a caller workspace.  Its counts,
offsets and gather / scatter indices must equal the workspace entry point's
bit for bit (the permutation's own tolerance), on consecutive calls that
share the static array.

This file is named to be collected last.
"""
import numpy as np
import pytest
import torch

from token_routing_expert_gb300 import native

pytestmark = pytest.mark.gpu


def _indices(T, k, E, seed):
    g = np.random.default_rng(seed)
    p = 1.0 / np.arange(1, E + 1)            # skewed load, some experts empty
    idx = g.choice(E, size=(T, k), p=p / p.sum())
    return torch.from_numpy(idx.astype(np.int32)).cuda()


@pytest.mark.parametrize("calls", [[(40000, 8, 896, 1), (3000, 4, 64, 2)], [(700, 2, 8, 3), (9000, 8, 1024, 4)]])
def test_noalloc_matches_workspace_permute_on_consecutive_calls(calls):
    for T, k, E, seed in calls:
        cfg = native.make_config(64, E, k, 64)
        idx = _indices(T, k, E, seed)
        ws = native.workspace(cfg, T)
        want = native.moe_permute(cfg, idx, ws)
        R = T * k
        got = (torch.full((E,), -7, dtype=torch.int32, device="cuda"),
               torch.full((E + 1,), -7, dtype=torch.int32, device="cuda"),
               torch.full((R,), -7, dtype=torch.int32, device="cuda"),
               torch.full((R,), -7, dtype=torch.int32, device="cuda"))
        native.moe_permute_noalloc(cfg, idx, *got)
        assert native.moe_get_status() == 0
        for a, b in zip(got, want):
            assert torch.equal(a, b)


def test_noalloc_rejects_calls_beyond_its_scratch():
    cfg = native.make_config(64, 1024, 8, 64)
    T = 300_000                                  # ceil(2.4M / 4096) * 1024 > 2^19 histogram entries
    idx = torch.zeros((T, 8), dtype=torch.int32, device="cuda")
    outs = (torch.empty(1024, dtype=torch.int32, device="cuda"), torch.empty(1025, dtype=torch.int32, device="cuda"),
            torch.empty(T * 8, dtype=torch.int32, device="cuda"), torch.empty(T * 8, dtype=torch.int32, device="cuda"))
    with pytest.raises(native.MoEError) as e:
        native.moe_permute_noalloc(cfg, idx, *outs)
    assert e.value.code == 2                     # MOE_ERR_UNSUPPORTED, nothing enqueued
    assert native.moe_get_status() == 0
