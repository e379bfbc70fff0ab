"""Prefix cache end to end on the GPU: a request that starts with a cached
system prompt reuses the blocks an earlier request filled, appends only the
rest, and its decode equals the oracle's attention over its own K/V.

K and V of a token are a fixed function of (token id, position) -- what a
model's layer would produce for the same prefix -- so reused blocks must hold
exactly the values the new request would have written itself."""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_154_gb300 as pa
from paged_kv_cache_154_gb300.engine import PagedKVCache

pytestmark = pytest.mark.gpu

H, HKV, D = 16, 4, 128


@pytest.fixture(scope="module", autouse=True)
def built():
    from paged_kv_cache_154_gb300 import build
    build.build()
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"


def kv_of(tokens, start):
    """[n, HKV, D] bf16 K and V for tokens at positions start, start + 1, ..."""
    k = np.stack([np.random.default_rng([int(t), start + i, 1]).standard_normal((HKV, D))
                  for i, t in enumerate(tokens)])
    v = np.stack([np.random.default_rng([int(t), start + i, 2]).standard_normal((HKV, D))
                  for i, t in enumerate(tokens)])
    return (torch.from_numpy(k).float().to(torch.bfloat16),
            torch.from_numpy(v).float().to(torch.bfloat16))


def serve(cache, tokens):
    """Admit a request: reuse cached blocks, append (and write) the rest."""
    seq, n = cache.pool.create_with_prefix(tokens)
    slots, pair = cache.pool.append_tokens(seq, tokens[n:])
    assert pair is None
    k, v = kv_of(tokens[n:], n)
    pa.append_kv(k.cuda(), v.cuda(), cache.k, cache.v,
                 torch.from_numpy(slots).cuda(), cache.num_blocks)
    return seq, n


def test_second_request_reuses_the_system_prompt_blocks():
    rng = np.random.default_rng(3)
    system = rng.integers(0, 32000, size=200).tolist()
    cache = PagedKVCache(64, HKV, D, "bf16")
    cache.pool.enable_prefix_cache(16)
    a_tokens = system + rng.integers(0, 32000, size=20).tolist()
    a, na = serve(cache, a_tokens)
    assert na == 0
    cache.pool.seq_free(a)                              # its full blocks stay cached
    b_tokens = system + rng.integers(0, 32000, size=37).tolist()
    b, nb = serve(cache, b_tokens)
    assert nb == 192                                    # 12 whole blocks of the prompt
    cached, registered, hits, lookups = cache.pool.prefix_stats()
    assert hits == 12
    # decode B's last token against its whole context
    L = len(b_tokens)
    bt, cl = cache.pool.block_tables([b], (L + 15) // 16)
    q = torch.randn(1, H, D, generator=torch.Generator().manual_seed(9)).to(torch.bfloat16)
    out = torch.empty(1, H, D, dtype=torch.float32, device="cuda")
    ws = torch.zeros(pa.decode_workspace_size(1, 1, H, HKV, D, 1, L), dtype=torch.uint8,
                     device="cuda")
    pa.decode(out, q.cuda(), cache.k, cache.v, torch.from_numpy(bt).cuda(),
              torch.from_numpy(cl).cuda(), L, 1.0 / np.sqrt(D), num_blocks=cache.num_blocks,
              workspace=ws)
    torch.cuda.synchronize()
    assert (code := pa.device_error()) == 0, hex(code)
    # the cache, read back, holds B's own K/V at B's positions (reused blocks included)
    host = oracle.empty_cache("bf16", cache.num_blocks, HKV, 16, D)
    host.k[...] = cache.k.view(torch.int16).cpu().numpy().view(np.uint16)
    host.v[...] = cache.v.view(torch.int16).cpu().numpy().view(np.uint16)
    k_ref, v_ref = kv_of(b_tokens, 0)
    t = np.arange(L)
    got_k = host.k[bt[0, t // 16], :, t % 16, :]
    assert np.array_equal(got_k, k_ref.view(torch.int16).numpy().view(np.uint16))
    got_v = host.v[bt[0, t // 16], :, t % 16, :]
    assert np.array_equal(got_v, v_ref.view(torch.int16).numpy().view(np.uint16))
    o, _, _ = oracle.attend(q.double().numpy(), host, bt, cl, None, H,
                            float(np.float32(1.0 / np.sqrt(D))))
    assert np.abs(out.double().cpu().numpy() - o).max() <= 2e-3
