"""Pins of the oracle's ZeRO-3 pieces: the per-layer gather and the peak ledger.

* Gathering every layer's range from the owners' BF16 shards and
  concatenating them gives back the full view the ZeRO-1/2 step all-gathers
  (all-gather assembles the shards into the full view: the ledger page, "one
  full ZeRO-3 computation"), bit for bit.
* Brute force: each gathered element is the one at its flat index in the
  concatenation of the shards.
* The peak ledger is the persistent ZeRO-3 subtotal (RC-T2 note N47: 32 GB
  for 8e9 parameters on 4 ranks) plus the live views.  A simulation of the
  two-slot schedule counts the bytes alive at every point and finds the same
  maximum.
"""
import numpy as np
import pytest


def test_layers_gathered_from_shards_rebuild_the_full_view(oracle_mod):
    rng = np.random.default_rng(0)
    sizes = [1000, 7, 3072, 768, 129, 4096]
    N = 4
    offsets, psi, psi_pad, shard = oracle_mod.layout(sizes, N)
    master = np.zeros(psi_pad, np.float32)
    master[:psi] = rng.standard_normal(psi) * 0.02
    m, v, w = np.zeros_like(master), np.zeros_like(master), np.zeros(psi_pad, np.uint16)
    grads = []
    for _ in range(N):
        g = np.zeros(psi_pad, np.float32)
        g[:psi] = rng.standard_normal(psi) * 1e-3
        grads.append(oracle_mod.f32_to_bf16(g))
    oracle_mod.zero_step(grads, master, m, v, w, oracle_mod.Hparams(), 1)
    shards = [w[r * shard:(r + 1) * shard].copy() for r in range(N)]
    parts = [oracle_mod.gather_range(shards, int(o), int(o) + n) for o, n in zip(offsets, sizes)]
    assert np.array_equal(np.concatenate(parts), w[:psi])
    assert np.array_equal(oracle_mod.gather_range(shards, 0, psi_pad), w)


@pytest.mark.parametrize("N,shard", [(1, 128), (3, 256), (8, 128)])
def test_gather_brute_force(oracle_mod, N, shard):
    rng = np.random.default_rng(N)
    shards = [rng.integers(0, 1 << 16, size=shard).astype(np.uint16) for _ in range(N)]
    full = np.concatenate(shards)
    for begin, end in [(0, 1), (5, 300), (shard - 3, shard + 3), (0, N * shard), (N * shard, N * shard)]:
        if end > N * shard:
            continue
        assert np.array_equal(oracle_mod.gather_range(shards, begin, end), full[begin:end])
    with pytest.raises(ValueError):
        oracle_mod.gather_range(shards, 0, N * shard + 1)


def test_peak_ledger_printed_persistent_part(oracle_mod):
    # with no layer gathered, the persistent ZeRO-3 subtotal: 32 GB for 8e9 on 4 ranks
    assert oracle_mod.zero3_peak_bytes([], 4) == 0
    assert oracle_mod.zero3_peak_bytes([8_000_000_000], 4) - 2 * 8_000_000_000 == 32_000_000_000


def _simulate_two_slot_peak(layers, N, g=2, o=12):
    """Walk the schedule: before layer i runs, layer i + 1 is prefetched into
    the other view; layer i's view is released once it ran.  Returns the most
    bytes alive at any point."""
    psi = sum(layers)
    persistent = (2 + g + o) * (-(-psi // N))
    live, peak = {}, persistent
    for i in range(len(layers)):
        live[i] = layers[i]                       # gathered (prefetched earlier)
        if i + 1 < len(layers):
            live[i + 1] = layers[i + 1]           # prefetch of the next layer
        peak = max(peak, persistent + 2 * sum(live.values()))
        del live[i]                               # released after use
    return peak


@pytest.mark.parametrize("layers", [[5, 9, 3, 9], [100], [7, 7, 7, 7, 7], [1, 1000, 1, 1000],
                                    [1000, 1, 1, 999], [3, 4]])
@pytest.mark.parametrize("N", [1, 4, 8])
def test_peak_ledger_matches_a_schedule_simulation(oracle_mod, layers, N):
    assert oracle_mod.zero3_peak_bytes(layers, N) == _simulate_two_slot_peak(layers, N)
