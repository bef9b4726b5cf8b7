"""GPU parity of the ZeRO-3 per-layer gather against the oracle.

* zero3_gather on ranges at aligned and odd offsets, across shard
  boundaries, with the tail and the whole vector.  The shards are separate
  buffers here.  The result must match the oracle's gather bit for bit.
* End to end: an in-place step writes the owners' BF16 shards (slices of the
  working-weight buffer).  Every layer of the GPT-2-small tensor list is then
  gathered with the two-view prefetch schedule and compared with the oracle's
  step and gather.
* The same schedule captured as a CUDA graph and replayed twice over
  different shard contents.
Both schedules run with one side stream (each gather chained to the one
before) and with two (neighbouring layers' gathers concurrent).
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("N,shard", [(1, 1024), (4, 65536), (8, 131072)])
def test_gather_ranges(zero_lib, oracle_mod, N, shard):
    Z = zero_lib
    dev = torch.device("cuda:0")
    rng = np.random.default_rng(N)
    host = [rng.integers(0, 1 << 16, size=shard).astype(np.uint16) for _ in range(N)]
    shards = [torch.from_numpy(h.view(np.int16).copy()).to(dev) for h in host]
    total = N * shard
    cases = [(0, total), (0, 8), (8, 24), (3, 3 + 1000), (shard - 13, min(total, shard + 29)),
             (total - 5, total), (16, 16 + 8 * 1234 + 5), (7, 7), (1, total - 1)]
    for b, e in cases:
        if e > total:
            assert Z.zero3_gather(shards, N, shard, b, e, shards[0], None) == Z.ZERO_ERR_ARG
            continue
        view = torch.full((max(e - b, 1) + 8,), -1, dtype=torch.int16, device=dev)
        assert Z.zero3_gather(shards, N, shard, b, e, view, None) == Z.ZERO_OK
        torch.cuda.synchronize()
        got = view.cpu().numpy().view(np.uint16)
        want = oracle_mod.gather_range(host, b, e)
        assert np.array_equal(got[:e - b], want), (b, e)
        assert (got[e - b:] == 0xFFFF).all(), "wrote past the range"


@pytest.mark.parametrize("side_streams", [1, 2])
def test_two_view_schedule_after_a_step(zero_lib, oracle_mod, side_streams):
    from zero_sharded_mixed_04_gb300 import synth
    from zero_sharded_mixed_04_gb300.optim import ZeroAdam, Zero3Views
    dev = torch.device("cuda:0")
    N = 4
    sizes = synth.gpt2_small_tensor_sizes()
    # layers: the embedding, then each block's ten tensors, then the final norm
    rc, lay, offs = zero_lib.zero_init_layout(sizes, N)
    assert rc == 0
    bounds = [0, 1] + [1 + 10 * (i + 1) for i in range(12)] + [len(sizes)]
    layers = [(offs[bounds[i]], offs[bounds[i + 1] - 1] + sizes[bounds[i + 1] - 1])
              for i in range(len(bounds) - 1)]
    assert layers[-1][1] == lay.psi
    psi, psi_pad, S = lay.psi, lay.psi_pad, lay.shard
    gen = torch.Generator().manual_seed(3)
    master = torch.zeros(psi_pad)
    master[:psi] = torch.randn(psi, generator=gen) * 0.02
    grads = []
    for _ in range(N):
        z = torch.zeros(psi_pad)
        z[:psi] = torch.randn(psi, generator=gen) * 1e-3
        grads.append(z.to(torch.bfloat16))
    opt = ZeroAdam(psi_pad, N, "bf16", weight_decay=0.1, device=dev, master=master.to(dev))
    opt.step([g.to(dev) for g in grads])
    w = opt.state()["w"]
    shards = [w[r * S:(r + 1) * S] for r in range(N)]
    got = {}

    def use(i, view):
        got[i] = view.clone()

    Zero3Views(shards, S, layers, device=dev, side_streams=side_streams).run(use)
    torch.cuda.synchronize()
    ref = {"master": master.numpy().copy(), "m": np.zeros(psi_pad, np.float32),
           "v": np.zeros(psi_pad, np.float32), "w": np.zeros(psi_pad, np.uint16)}
    oracle_mod.zero_step([g.view(torch.int16).numpy().view(np.uint16) for g in grads],
                         ref["master"], ref["m"], ref["v"], ref["w"],
                         oracle_mod.Hparams(weight_decay=0.1), 1)
    oshards = [ref["w"][r * S:(r + 1) * S] for r in range(N)]
    for i, (b, e) in enumerate(layers):
        want = oracle_mod.gather_range(oshards, b, e)
        assert np.array_equal(got[i].cpu().numpy().view(np.uint16), want), f"layer {i}"


@pytest.mark.parametrize("side_streams", [1, 2])
def test_two_view_schedule_as_a_cuda_graph(zero_lib, oracle_mod, side_streams):
    """The two-view pass captured once and replayed: each replay gathers what
    the shards hold at that moment, like the eager pass."""
    from zero_sharded_mixed_04_gb300 import synth
    from zero_sharded_mixed_04_gb300.optim import Zero3Views
    dev = torch.device("cuda:0")
    N = 4
    sizes = synth.gpt2_small_tensor_sizes()
    rc, lay, offs = zero_lib.zero_init_layout(sizes, N)
    assert rc == 0
    bounds = [0, 1] + [1 + 10 * (i + 1) for i in range(12)] + [len(sizes)]
    layers = [(offs[bounds[i]], offs[bounds[i + 1] - 1] + sizes[bounds[i + 1] - 1])
              for i in range(len(bounds) - 1)]
    S = lay.shard
    w = torch.empty(lay.psi_pad, dtype=torch.int16, device=dev)
    shards = [w[r * S:(r + 1) * S] for r in range(N)]
    outs = [torch.empty(e - b, dtype=torch.int16, device=dev) for b, e in layers]

    def use(i, view):
        outs[i].copy_(view)

    views = Zero3Views(shards, S, layers, device=dev, side_streams=side_streams)
    graph = views.capture(use)
    for seed in (41, 42):
        host = torch.randint(-32768, 32767, (lay.psi_pad,), dtype=torch.int16,
                             generator=torch.Generator().manual_seed(seed))
        w.copy_(host)
        for o in outs:
            o.fill_(0x5A5A)
        graph.replay()
        torch.cuda.synchronize()
        hs = host.numpy().view(np.uint16)
        oshards = [hs[r * S:(r + 1) * S] for r in range(N)]
        for i, (b, e) in enumerate(layers):
            want = oracle_mod.gather_range(oshards, b, e)
            assert np.array_equal(outs[i].cpu().numpy().view(np.uint16), want), f"seed {seed} layer {i}"


def test_overlapping_gathers_into_distinct_views(zero_lib, oracle_mod):
    """Consecutive gathers launched with ZERO3_GATHER_OVERLAP_PREVIOUS into
    separate views (none touches another's view, all only read the shards):
    each may start while the previous drains, and every view must still equal
    the oracle's gather."""
    Z = zero_lib
    dev = torch.device("cuda:0")
    N, shard = 8, 131072
    rng = np.random.default_rng(77)
    host = [rng.integers(0, 1 << 16, size=shard).astype(np.uint16) for _ in range(N)]
    shards = [torch.from_numpy(h.view(np.int16).copy()).to(dev) for h in host]
    total = N * shard
    bounds = [0, 40_000, 40_008, 300_016, 300_021, 700_000, 1_000_003, total]
    layers = list(zip(bounds[:-1], bounds[1:]))
    views = [torch.full((e - b + 8,), -1, dtype=torch.int16, device=dev) for b, e in layers]
    for _ in range(3):
        for i, ((b, e), v) in enumerate(zip(layers, views)):
            flags = Z.ZERO3_GATHER_OVERLAP_PREVIOUS if i else 0
            assert Z.zero3_gather(shards, N, shard, b, e, v, None, flags=flags) == Z.ZERO_OK
    torch.cuda.synchronize()
    for (b, e), v in zip(layers, views):
        got = v.cpu().numpy().view(np.uint16)
        assert np.array_equal(got[:e - b], oracle_mod.gather_range(host, b, e)), (b, e)
        assert (got[e - b:] == 0xFFFF).all(), "wrote past the range"
