"""moe_permute_noalloc against the oracle's permutation and against moe_permute.

Some callers may not allocate device memory at all: a serving loop that gave
all of it to its own pool at start-up, or a plug-in host that only hands a
library its input and output buffers.  moe_permute_noalloc serves them with
a fixed static scratch array instead of a caller workspace.  Its counts,
offsets and gather / scatter indices must equal the oracle's counting sort
and the workspace entry point's bit for bit (the permutation's own
tolerance), on consecutive calls that share the static array: both calls of
a pair take the multi-pass path that uses the array (more than 16,384
assignments), the first with more chunks and experts than the second, so
stale histogram entries of the first call lie inside the second's range of
the array.

This file is named to be collected last.
"""
import numpy as np
import pytest
import torch

from oracle import moe_ref as ref
from token_routing_expert_gb300 import native

pytestmark = pytest.mark.gpu


def _indices(T, k, E, seed):
    g = np.random.default_rng(seed)
    p = 1.0 / np.arange(1, E + 1)            # skewed load, some experts empty
    idx = g.choice(E, size=(T, k), p=p / p.sum())
    return idx.astype(np.int32)


def _outputs(E, R):
    # filled with a value no result takes, so an entry the call leaves unwritten shows
    return (torch.full((E,), -7, dtype=torch.int32, device="cuda"),
            torch.full((E + 1,), -7, dtype=torch.int32, device="cuda"),
            torch.full((max(R, 1),), -7, dtype=torch.int32, device="cuda"),
            torch.full((max(R, 1),), -7, dtype=torch.int32, device="cuda"))


def _check(got, idx_np, E, cfg, idx):
    R = idx_np.size
    p = ref.permute(idx_np.astype(np.int64), E)
    np.testing.assert_array_equal(got[0].cpu().numpy(), p.counts)
    np.testing.assert_array_equal(got[1].cpu().numpy(), p.offsets)
    np.testing.assert_array_equal(got[2][:R].cpu().numpy(), p.gather_token)
    np.testing.assert_array_equal(got[3][:R].cpu().numpy(), p.scatter_pos)
    ws = native.workspace(cfg, idx.shape[0])
    want = native.moe_permute(cfg, idx, ws)
    for a, b in zip(got, want):
        assert torch.equal(a[:b.numel()], b)


@pytest.mark.parametrize("calls", [
    [(40000, 8, 896, 1), (5000, 4, 64, 2)],      # 320,000 then 20,000 assignments, both multi-pass
    [(9000, 8, 1024, 3), (40000, 8, 896, 4)],    # 72,000 then 320,000
    [(700, 2, 8, 5), (3000, 8, 256, 6)],         # the one-launch cluster path, then the array
])
def test_noalloc_matches_oracle_on_consecutive_calls(calls):
    for T, k, E, seed in calls:
        cfg = native.make_config(64, E, k, 64)
        idx_np = _indices(T, k, E, seed)
        idx = torch.from_numpy(idx_np).cuda()
        got = _outputs(E, T * k)
        native.moe_permute_noalloc(cfg, idx, *got)
        assert native.moe_get_status() == 0
        _check(got, idx_np, E, cfg, idx)


def test_noalloc_calls_on_two_streams_ordered_by_an_event():
    """The second call runs on another stream, after the first by an event (the caller's ordering);
    both use the array, and each result must be its own."""
    s1, s2 = torch.cuda.Stream(), torch.cuda.Stream()
    runs = []
    for (T, k, E, seed) in [(30000, 8, 512, 7), (6000, 4, 128, 8)]:
        cfg = native.make_config(64, E, k, 64)
        idx_np = _indices(T, k, E, seed)
        idx = torch.from_numpy(idx_np).cuda()
        runs.append((cfg, idx_np, idx, E, _outputs(E, T * k)))
    torch.cuda.synchronize()
    done = torch.cuda.Event()
    with torch.cuda.stream(s1):
        cfg, _, idx, _, got = runs[0]
        native.moe_permute_noalloc(cfg, idx, *got, stream=s1)
        done.record(s1)
    with torch.cuda.stream(s2):
        s2.wait_event(done)
        cfg, _, idx, _, got = runs[1]
        native.moe_permute_noalloc(cfg, idx, *got, stream=s2)
    torch.cuda.synchronize()
    assert native.moe_get_status() == 0
    for cfg, idx_np, idx, E, got in runs:
        _check(got, idx_np, E, cfg, idx)


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


def test_noalloc_wrapper_rejects_undersized_outputs():
    cfg = native.make_config(64, 16, 4, 64)
    idx = torch.zeros((100, 4), dtype=torch.int32, device="cuda")
    good = _outputs(16, 400)
    for i, short in enumerate((15, 16, 399, 399)):
        outs = list(good)
        outs[i] = torch.empty(short, dtype=torch.int32, device="cuda")
        with pytest.raises(ValueError):
            native.moe_permute_noalloc(cfg, idx, *outs)
    with pytest.raises(ValueError):
        native.moe_permute_noalloc(cfg, idx[:, :3].contiguous(), *good)
    assert native.moe_get_status() == 0
