"""Prefix reuse end to end on the GPU: requests that share a system prompt take
its blocks from the prefix cache, write K/V and run attention only for their
uncached remainder, and get the same rows as the fp64 oracle over their whole
context -- and, within rounding, the same rows as a run without the cache."""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_263_gb300 as pkv
from synth import normal_bf16, stream_key
from tests.gpu_util import TOL, bits, max_abs, require_gpu

pytestmark = pytest.mark.gpu

HQ, HKV, D, BS = 16, 2, 128, 16
SEED = 4242


@pytest.fixture(scope="module", autouse=True)
def gpu():
    require_gpu()


def _kv(tokens, pos, which):
    """K or V rows [len(pos)][HKV][D]: a function of (token id, position) only,
    as a model's K/V at a position depend only on the tokens up to it."""
    t = torch.as_tensor(np.asarray(tokens, dtype=np.int64))[:, None, None]
    p = torch.as_tensor(np.asarray(pos, dtype=np.int64))[:, None, None]
    h = torch.arange(HKV, dtype=torch.int64)[None, :, None]
    d = torch.arange(D, dtype=torch.int64)[None, None, :]
    ctr = ((t * 65536 + p) * HKV + h) * D + d
    return normal_bf16(stream_key(SEED, which), ctr)


def _q(req, n):
    ctr = torch.arange(n * HQ * D, dtype=torch.int64).reshape(n, HQ, D)
    return normal_bf16(stream_key(SEED, 100 + req), ctr)


class _Server:
    """Minimal scheduler around the library: pool, prefix cache, paged caches."""

    def __init__(self, num_blocks, use_cache, seed):
        order = np.random.default_rng(seed).permutation(num_blocks).astype(np.int32)
        self.pool = pkv.KVPool(num_blocks, order)
        self.cache = pkv.PrefixCache(self.pool) if use_cache else None
        # every slot starts as NaN: anything read that was never written shows
        self.k = torch.full((num_blocks, HKV, BS, D), float("nan"), dtype=torch.bfloat16, device="cuda")
        self.v = torch.full_like(self.k, float("nan"))

    def run(self, reqs):
        """reqs: list of (req id, tokens).  One mixed call for the batch; returns
        per request (first computed position, output rows [n][HQ][D])."""
        tables, starts = [], []
        for _, toks in reqs:
            nblk = -(-len(toks) // BS)
            # leave the last token to compute, as a real request must
            hit = self.cache.match(toks[:-1]) if self.cache else np.zeros(0, np.int32)
            own = self.cache.alloc(nblk - len(hit)) if self.cache else self.pool.alloc(nblk)
            tables.append(np.concatenate([hit, own]).astype(np.int32))
            starts.append(BS * len(hit))
        mb = max(len(t) for t in tables)
        bt = np.full((len(reqs), mb), -1, np.int32)
        for i, t in enumerate(tables):
            bt[i, :len(t)] = t
        qs, slots, ks, vs, cu = [], [], [], [], [0]
        for (rid, toks), t, s in zip(reqs, tables, starts):
            pos = np.arange(s, len(toks))
            ks.append(_kv(np.asarray(toks)[pos], pos, 1))
            vs.append(_kv(np.asarray(toks)[pos], pos, 2))
            slots.append(t[pos // BS].astype(np.int64) * BS + pos % BS)
            qs.append(_q(rid, len(toks))[s:])
            cu.append(cu[-1] + len(pos))
        dev = "cuda"
        pkv.reshape_and_cache(torch.cat(ks).to(dev), torch.cat(vs).to(dev), self.k, self.v,
                              torch.as_tensor(np.concatenate(slots)).to(dev))
        q = torch.cat(qs).to(dev)
        out = torch.empty(q.shape, dtype=torch.float32, device=dev)
        lens = torch.as_tensor([len(t) for _, t in reqs], dtype=torch.int32, device=dev)
        pkv.paged_attention_chunked_prefill(out, q, torch.as_tensor(cu, dtype=torch.int32, device=dev), lens,
                                            max(np.diff(cu)), self.k, self.v, torch.as_tensor(bt).to(dev))
        assert pkv.kv_last_device_status() == 0, pkv.kv_last_device_status_flags()
        res = out.cpu().numpy().astype(np.float64)
        for (rid, toks), t in zip(reqs, tables):
            if self.cache:
                self.cache.insert(toks, t)
            self.pool.free(t)
        return [(s, res[cu[i]:cu[i + 1]]) for i, s in enumerate(starts)]


def _expected(rid, toks, start):
    pos = np.arange(len(toks))
    k = oracle.bf16_bits_to_f64(bits(_kv(toks, pos, 1)))
    v = oracle.bf16_bits_to_f64(bits(_kv(toks, pos, 2)))
    q = oracle.bf16_bits_to_f64(bits(_q(rid, len(toks))[start:]))
    return oracle.contiguous_attention(q, k, v)


def test_shared_system_prompt_is_prefilled_once():
    rng = np.random.default_rng(5)
    sys_prompt = [int(x) for x in rng.integers(0, 50000, size=2000)]
    reqs = [(r, sys_prompt + [int(x) for x in rng.integers(0, 50000, size=n)])
            for r, n in enumerate([100, 300, 37, 1])]
    srv = _Server(1200, True, 1)
    first = srv.run(reqs[:1])
    assert first[0][0] == 0
    batch = srv.run(reqs[1:])
    # each later request reuses the 125 blocks of the prompt and computes the rest
    assert [s for s, _ in batch] == [2000, 2000, 2000]
    st = srv.cache.stats()
    assert st["hit_blocks"] == 3 * 125 and st["cached_blocks"] == 125 + sum((len(t) // BS) - 125 for _, t in reqs)
    for (rid, toks), (s, rows) in zip(reqs, first + batch):
        err = max_abs(rows, _expected(rid, toks, s))
        assert err <= TOL["bf16"], (rid, err)
    # without the cache every request prefills its whole prompt; the rows agree
    # with the cached run's within rounding.  They are not bitwise equal: the
    # chunk kernel's KV partitions follow the batch shape (its wave model), so
    # a 300-row chunk and a 2,300-row prompt cut the same keys differently.
    plain = _Server(1200, False, 2)
    for (rid, toks), (s, rows) in zip(reqs[1:], batch):
        (_, full), = plain.run([(rid, toks)])
        assert max_abs(full[s:], rows) <= TOL["bf16"], rid


def test_tenant_keys_keep_prefixes_apart_on_the_gpu():
    rng = np.random.default_rng(6)
    prompt = [int(x) for x in rng.integers(0, 50000, size=640)]
    srv = _Server(400, True, 3)
    srv.run([(0, prompt + [7])])
    tb = srv.cache.match(prompt, salt=99)
    assert tb.size == 0
    (s, rows), = srv.run([(1, prompt + [8, 9])])
    assert s == 640
    assert max_abs(rows, _expected(1, prompt + [8, 9], s)) <= TOL["bf16"]
