"""Read-once shared-prefix decode (pa_decode_shared_prefix) vs the CPU
oracle: forks of one prompt read their shared blocks once per group, and the
result must still be the plain attention of every fork (within 2e-3 for
16-bit caches, fp32 output)."""
import os

import numpy as np
import pytest
import torch

import oracle
import workloads as W
import paged_kv_cache_154_gb300 as pa
from gpu_harness import THREADS, check_cache_bits, check_out, run_both

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    from paged_kv_cache_154_gb300 import build
    build.build()
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"


CASES = {
    # GQA 4, d 64, fp16: 3 prompts x 4 forks
    "gqa4_f16_d64": lambda: W.best_of_n("sp_gqa4", 71, num_groups=3, n_forks=4, prompt_len=200,
                                        shared_extra_max=15, private_max=40, num_heads=8,
                                        num_kv_heads=2, head_dim=64, kv_dtype="f16"),
    # GQA 8, d 128, verify runs of 1-5 inside the groups: up to 120 rows per group
    "gqa8_verify": lambda: W.best_of_n("sp_verify", 72, num_groups=2, n_forks=3,
                                       prompt_len=300, shared_extra_max=9, private_max=60,
                                       num_heads=16, num_kv_heads=2, head_dim=128,
                                       step_q_max=5),
    # MQA 32 q heads: 5 forks give 160 rows per KV head (5 row chunks)
    "mqa32_5forks": lambda: W.best_of_n("sp_mqa", 73, num_groups=2, n_forks=5, prompt_len=500,
                                        shared_extra_max=15, private_max=100, num_heads=32,
                                        num_kv_heads=1, head_dim=128),
    # groups of one: no prefix phase work, every sequence in the suffix phase
    "singletons": lambda: W.best_of_n("sp_single", 74, num_groups=5, n_forks=1,
                                      prompt_len=130, shared_extra_max=15, private_max=50,
                                      num_heads=8, num_kv_heads=2, head_dim=64),
    # long prompts, 4 forks x GQA 4 = 16 rows per KV head: the prefix phase
    # runs the per-warp kernel with its in-kernel merge (8 blocks per worker
    # and more), writing the base-2 log-sum-exps the final merge needs
    "long_prefix_in_kernel": lambda: W.best_of_n("sp_long", 76, num_groups=8, n_forks=4,
                                                 prompt_len=4096, shared_extra_max=15,
                                                 private_max=64, num_heads=32, num_kv_heads=8,
                                                 head_dim=128),
    # 16-bit caches with d 128 and 17-64 rows per (group, kv head) over long
    # prefixes take the tensor-core prefix phase: key chunks of each (group,
    # kv head) in two streams per CTA, merged per row afterwards. Prefixes of
    # 1,100-2,000 tokens: one chunk pair, some groups with one chunk only;
    # fp16, verify runs of 1-2 (24-48 rows)
    "tc_prefix_ragged": lambda: W.best_of_n("sp_tc_ragged", 77, num_groups=3, n_forks=3,
                                            prompt_len=1100, shared_extra_max=900,
                                            private_max=40, num_heads=16, num_kv_heads=2,
                                            head_dim=128, kv_dtype="f16", step_q_max=2),
    # 4,096-token prefixes over 16 (group, kv head) tasks: four chunk pairs each
    "tc_prefix_chunks": lambda: W.best_of_n("sp_tc_chunks", 78, num_groups=8, n_forks=5,
                                            prompt_len=4096, shared_extra_max=15,
                                            private_max=64, num_heads=16, num_kv_heads=2,
                                            head_dim=128),
    # a prompt that fills its last block: forks share every prompt block
    "block_aligned_prompt": lambda: W.best_of_n("sp_aligned", 75, num_groups=2, n_forks=3,
                                                prompt_len=255, shared_extra_max=1,
                                                private_max=0, num_heads=8, num_kv_heads=2,
                                                head_dim=128),
}


@pytest.mark.parametrize("name", list(CASES))
def test_shared_prefix_matches_oracle(name):
    wl = CASES[name]()
    ref, cache, si, out = run_both(wl, shared_prefix=True)
    check_cache_bits(ref, cache)
    check_out(ref, out, wl.kv_dtype)
    sp = si.shared
    if name == "singletons":
        assert (sp.prefix_len_host == 0).all()
    else:
        assert (sp.prefix_len_host >= 128).all()     # the groups really share blocks


def test_best_of_5_config_read_once():
    wl = W.llama2_70b_best_of_5()
    ref, cache, si, out = run_both(wl, shared_prefix=True)
    check_out(ref, out, wl.kv_dtype)
    assert len(si.shared.prefix_len_host) == 8 and (si.shared.prefix_len_host == 4096).all()


def test_shared_prefix_output_in_q_dtype():
    wl = CASES["gqa8_verify"]()
    ref, cache, si, out = run_both(wl, out_dtype=torch.bfloat16, shared_prefix=True)
    check_out(ref, out, wl.kv_dtype, torch.bfloat16)


def _tiny_state():
    wl = W.tiny()
    ref, cache, si, _ = run_both(wl)
    return wl, ref, cache, si


def test_raw_api_prefix_covering_a_whole_sequence():
    """Two query sets against the same sequence (same block table, L = 64):
    their group's prefix is all 64 tokens, so the suffix phase attends
    nothing for them; a third sequence forms a group of one."""
    wl, ref, cache, si = _tiny_state()
    bt = si.block_tables.cpu().numpy()
    cl = si.context_lens.cpu().numpy()
    pick = [2, 2, 3]                                   # L = 64, 64, 100
    assert cl[2] == 64
    bt2, cl2 = bt[pick], cl[pick]
    g = torch.Generator().manual_seed(5)
    q = torch.randn(3, wl.num_heads, wl.head_dim, generator=g).to(torch.float16)
    gs = np.array([0, 2, 3], np.int32)
    pl = np.array([64, 0], np.int32)
    dev = "cuda"
    out = torch.empty(3, wl.num_heads, wl.head_dim, dtype=torch.float32, device=dev)
    ws = torch.zeros(pa.decode_shared_prefix_workspace_size(3, 3, wl.num_heads, wl.num_kv_heads,
                                                            wl.head_dim, 1, 100, 2, 2, 64,
                                                            bt.shape[1]),
                     dtype=torch.uint8, device=dev)
    pa.decode_shared_prefix(out, q.to(dev), cache.k, cache.v, torch.from_numpy(bt2).to(dev),
                            torch.from_numpy(cl2).to(dev), 100, wl.scale,
                            torch.from_numpy(gs).to(dev), torch.from_numpy(pl).to(dev), 2, 64,
                            num_blocks=cache.num_blocks, workspace=ws)
    torch.cuda.synchronize()
    assert (code := pa.device_error()) == 0, hex(code)
    o, _, _ = oracle.attend(q.double().numpy(), ref.cache, bt2, cl2, None, wl.num_heads,
                            wl.scale)
    assert np.abs(out.double().cpu().numpy() - o).max() <= 2e-3


def test_validate_mode_rejects_inconsistent_groups(monkeypatch):
    wl, ref, cache, si = _tiny_state()
    monkeypatch.setenv("PA_VALIDATE", "1")
    dev = "cuda"
    bt = si.block_tables
    cl = si.context_lens
    out = torch.empty_like(si.out)
    ws = torch.zeros(pa.decode_shared_prefix_workspace_size(4, 4, wl.num_heads, wl.num_kv_heads,
                                                            wl.head_dim, 1, 100, 4, 4, 96,
                                                            bt.shape[1]),
                     dtype=torch.uint8, device=dev)

    def call(gs, pl, max_prefix=96):
        pa.decode_shared_prefix(out, si.q, cache.k, cache.v, bt, cl, 100, wl.scale,
                                torch.tensor(gs, dtype=torch.int32, device=dev),
                                torch.tensor(pl, dtype=torch.int32, device=dev), 4, max_prefix,
                                num_blocks=cache.num_blocks, workspace=ws)

    for gs, pl in ([[0, 4], [16]],          # the four sequences hold different blocks
                   [[0, 1, 4], [32, 0]],    # 32 tokens reach the query of a 17-token sequence
                   [[0, 2, 4], [8, 0]],     # not a whole block
                   [[0, 3], [0]]):          # groups do not cover the batch
        with pytest.raises(pa.PAError) as e:
            call(gs, pl)
        assert e.value.status == 6
    call([0, 1, 2, 3, 4], [0, 0, 0, 0])     # consistent: accepted
    torch.cuda.synchronize()
    assert np.abs(out.double().cpu().numpy() - ref.out).max() <= 2e-3


def test_shared_prefix_graph_replay_matches_eager():
    wl = CASES["gqa4_f16_d64"]()
    ref, cache, si, out = run_both(wl, shared_prefix=True)
    eager = out.clone()
    g = cache.capture(cache.attend_step, si, wl.scale)
    si.out.zero_()
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(si.out, eager)
