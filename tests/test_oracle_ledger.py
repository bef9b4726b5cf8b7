"""Pins of the oracle's memory ledger, communication count and flat layout
against the numbers the pages print (tests/golden/*.txt, each line cited) and
against brute force."""
import os

import pytest

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _rows(name):
    rows = []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            data, cite = line.split("|", 1)
            rows.append(([int(x) for x in data.split()], cite.strip()))
    return rows


@pytest.mark.parametrize("row", _rows("ledger_pages.txt"), ids=lambda r: r[1][:40])
def test_ledger_printed_values(oracle_mod, row):
    (psi, N, stage, g, o, expected), cite = row
    assert oracle_mod.ledger_bytes(psi, N, stage, g, o) == expected, cite


@pytest.mark.parametrize("row", _rows("stage_table.txt"), ids=lambda r: r[1][:30])
@pytest.mark.parametrize("N", [1, 2, 3, 4, 8, 64])
def test_stage_table_per_param(oracle_mod, row, N):
    (stage, const, over_n, comm), cite = row
    psi = 1_000_003 * N  # divisible by N, so the closed form is exact
    # bytes per parameter = const + over_n / N
    assert oracle_mod.ledger_bytes(psi, N, stage) * N == (const * N + over_n) * psi, cite
    assert oracle_mod.comm_volume(psi, N, stage) == comm * psi, cite


def test_ledger_sharded_parts_round_up(oracle_mod):
    # psi not divisible by N: a sharded part holds ceil(psi/N) elements per rank
    psi, N = 10, 4
    assert oracle_mod.ledger_bytes(psi, N, 3) == 16 * 3
    assert oracle_mod.ledger_bytes(psi, N, 1) == 4 * 10 + 12 * 3
    assert oracle_mod.ledger_bytes(psi, N, 2) == 2 * 10 + 14 * 3
    assert oracle_mod.ledger_bytes(psi, N, 5) == -1


def _ring_send_count(psi, N, passes):
    """Brute force: simulate ring reduce-scatter / all-gather passes and count
    the elements every rank sends (N-1 hops per pass, one chunk per hop)."""
    chunk = [psi // N + (1 if r < psi % N else 0) for r in range(N)]
    sent = [0] * N
    for _ in range(passes):
        for hop in range(N - 1):
            for r in range(N):
                # in hop h rank r forwards the chunk index (r - h) mod N
                sent[r] += chunk[(r - hop) % N]
    return max(sent)


@pytest.mark.parametrize("psi", [1, 7, 1000, 1024])
@pytest.mark.parametrize("N", [1, 2, 3, 4, 8])
@pytest.mark.parametrize("stage", [0, 1, 2, 3])
def test_comm_volume_ring_brute_force(oracle_mod, psi, N, stage):
    passes = 3 if stage == 3 else 2
    # the largest rank sends at most (N-1) * ceil(psi/N) per pass
    assert oracle_mod.comm_volume(psi, N, stage, ring_exact=True) >= _ring_send_count(psi, N, passes)
    if psi % N == 0:
        assert oracle_mod.comm_volume(psi, N, stage, ring_exact=True) == _ring_send_count(psi, N, passes)


def test_comm_volume_ring_tends_to_page_count(oracle_mod):
    psi = 10**9
    for stage, mult in ((0, 2), (1, 2), (2, 2), (3, 3)):
        ring = oracle_mod.comm_volume(psi, 1024, stage, ring_exact=True)
        assert abs(ring / psi - mult) < mult / 1000


@pytest.mark.parametrize("numel,N", [([1], 1), ([3, 5, 7], 4), ([128] * 8, 8), ([1000, 24], 3), ([], 2),
                                     ([5], 7)])
def test_layout_brute_force(oracle_mod, numel, N):
    offsets, psi, psi_pad, shard = oracle_mod.layout(numel, N)
    assert psi == sum(numel)
    assert psi_pad % (N * 128) == 0 and psi <= psi_pad < psi + N * 128
    assert shard * N == psi_pad
    # prefix sums, no gaps, no overlaps
    pos = 0
    for i, n in enumerate(numel):
        assert offsets[i] == pos
        pos += n
    # every flat index belongs to exactly one owner's contiguous slice
    owner_of = [None] * psi_pad
    for r in range(N):
        for j in range(r * shard, (r + 1) * shard):
            assert owner_of[j] is None
            owner_of[j] = r
    assert all(o is not None for o in owner_of)


def test_layout_of_the_benchmark_workloads(oracle_mod):
    """Padded sizes of the five workloads: the flat vector is padded to a
    multiple of N*128 elements."""
    from zero_sharded_mixed_04_gb300 import synth
    expected = {"flat1m_n4": (1_048_576, 1_048_576), "gpt2small_n4": (123_588_864, 123_589_120),
                "flat1b_n8": (1_000_000_000, 1_000_000_512),
                "flat3b_n4_fp32": (3_000_000_000, 3_000_000_000),
                "ragged6b_n4": (6_000_000_007, 6_000_000_512)}
    for name, (psi, psi_pad) in expected.items():
        wl = synth.WORKLOADS[name]
        sizes = synth.ragged6b_tensor_sizes() if name == "ragged6b_n4" else wl.sizes
        _, p, pp, shard = oracle_mod.layout(sizes, wl.N)
        assert (p, pp) == (psi, psi_pad), name
        assert wl.psi == psi and wl.psi_pad == psi_pad
    sizes = synth.ragged6b_tensor_sizes()
    assert min(sizes) == 1 and max(sizes) == 1 << 27
