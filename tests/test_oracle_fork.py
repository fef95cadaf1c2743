"""Parallel sampling (n generations from one prompt) in the oracle's block
accounting: the prompt's blocks are shared by every sample, and the first write
of each sample into a shared block gives it its own copy ("M.65 Inference
serving", block management (g): initially share the prefix blocks, copy the
affected block when generations diverge; "Waste, and three ways to reclaim it",
"Copy on write")."""
import pytest

from oracle import model as omodel
from synth.workloads import small_workload


def _blocks(t):
    return -(-t // 16)


@pytest.mark.parametrize("prompt,gens", [(1000, [37, 1, 200, 64]), (1000, [5] * 8), (40, [1, 2, 3])])
def test_parallel_sampling_shares_the_prompt_and_copies_the_partial_block(prompt, gens):
    n = len(gens)
    lens = [prompt + g for g in gens]
    pb = _blocks(prompt)
    wl = small_workload(1300 + n, lens=lens, prefix_tokens=prompt, cow_block=pb - 1)
    tb = omodel.build_tables(wl)
    # the full prompt blocks are one physical copy held n times
    full = pb - 1
    for j in range(full):
        assert len(set(tb.tables[:, j].tolist())) == 1
        assert tb.pool.ref[int(tb.tables[0, j])] == n
    # the partial block: n - 1 samples got copies, the last writer keeps the original
    last = tb.tables[:, pb - 1]
    assert len(set(last.tolist())) == n
    assert len(tb.copies) == n - 1 and tb.pool.stats()["cow_copies"] == n - 1
    assert all(tb.pool.ref[int(b)] == 1 for b in last)
    # blocks in use, against n private copies of the prompt
    live = tb.pool.stats()["live"]
    assert live == full + n + sum(_blocks(L) - pb for L in lens)
    assert sum(_blocks(L) for L in lens) - live == (n - 1) * full


def test_block_aligned_prompt_needs_no_copy():
    """A prompt that ends on a block boundary: the samples' first tokens go to
    fresh blocks, so nothing is copied and every prompt block stays shared."""
    prompt, gens = 1008, [3, 40, 17]
    lens = [prompt + g for g in gens]
    wl = small_workload(1310, lens=lens, prefix_tokens=prompt)
    tb = omodel.build_tables(wl)
    assert tb.pool.stats()["cow_copies"] == 0
    for j in range(prompt // 16):
        assert tb.pool.ref[int(tb.tables[0, j])] == len(gens)
    assert tb.pool.stats()["live"] == prompt // 16 + sum(_blocks(L) - prompt // 16 for L in lens)
