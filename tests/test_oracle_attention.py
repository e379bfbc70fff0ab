"""Pins for the oracle's attention (CPU only).

Each test ties the oracle to something other than itself: a library routine
(torch scaled_dot_product_attention in fp64), a brute-force computation on
the contiguous K/V before paging, closed forms, and invariants the method
must satisfy. Plausible mistakes (a wrong GQA head map, an off-by-one causal
bound, a lost scale, a wrong gather) are planted on the CPU side and shown to
fail the pins.
"""
import dataclasses

import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle
import workloads as W


def sdpa_reference(wl, kv_list, gqa="interleave", causal_shift=0, scale=None):
    """fp64 torch SDPA per sequence with an explicit causal mask offset by L - r."""
    scale = wl.scale if scale is None else scale
    G = wl.num_heads // wl.num_kv_heads
    qsl = wl.query_start_loc
    outs = []
    for i, (K, V) in enumerate(kv_list):
        L = K.shape[0]
        q = wl.q[qsl[i]:qsl[i + 1]].double()                   # [r, H, d]
        r = q.shape[0]
        Kd = K.double().permute(1, 0, 2)                        # [Hkv, L, d]
        Vd = V.double().permute(1, 0, 2)
        if gqa == "interleave":
            Kd = Kd.repeat_interleave(G, 0)
            Vd = Vd.repeat_interleave(G, 0)
        else:                                                   # planted mistake: h % H_kv
            Kd = Kd.repeat(G, 1, 1)
            Vd = Vd.repeat(G, 1, 1)
        t = torch.arange(L)
        qi = torch.arange(r)
        mask = t[None, :] <= (L - r + qi[:, None] + causal_shift)   # [r, L]
        o = F.scaled_dot_product_attention(q.permute(1, 0, 2)[None], Kd[None], Vd[None],
                                           attn_mask=mask[None, None], scale=scale)
        outs.append(o[0].permute(1, 0, 2))                      # [r, H, d]
    return torch.cat(outs, 0).numpy()


def brute_force(wl, kv_list):
    """Naive loops over the contiguous data: logits, max, exp, weighted sum."""
    G = wl.num_heads // wl.num_kv_heads
    qsl = wl.query_start_loc
    out = np.zeros((qsl[-1], wl.num_heads, wl.head_dim))
    for s, (K, V) in enumerate(kv_list):
        K = K.double().numpy()
        V = V.double().numpy()
        L = K.shape[0]
        r = qsl[s + 1] - qsl[s]
        for i in range(r):
            vis = L - r + i + 1
            for h in range(wl.num_heads):
                qv = wl.q[qsl[s] + i, h].double().numpy()
                z = wl.scale * (K[:vis, h // G, :] @ qv)
                w = np.exp(z - z.max())
                out[qsl[s] + i, h] = (w @ V[:vis, h // G, :]) / w.sum()
    return out


def small_cases():
    return [
        W.tiny(),
        W.simple("gqa4_bf16", 11, [1, 15, 16, 17, 31, 48, 130], [1] * 7, 8, 2, 128, "bf16"),
        W.simple("mqa_verify", 12, [5, 40, 77, 96], [5, 2, 1, 4], 8, 1, 64, "bf16"),
        W.simple("mha_f16", 13, [33, 2, 64], [1, 2, 3], 4, 4, 64, "f16"),
    ]


@pytest.mark.parametrize("wl", small_cases(), ids=lambda w: w.name)
def test_matches_torch_sdpa_fp64(wl):
    run = oracle.run(wl)
    ref = sdpa_reference(wl, W.contiguous_kv(wl))
    np.testing.assert_allclose(run.out, ref, rtol=0, atol=1e-12)


@pytest.mark.parametrize("wl", small_cases()[:2], ids=lambda w: w.name)
def test_matches_brute_force_on_unpaged_data(wl):
    run = oracle.run(wl)
    ref = brute_force(wl, W.contiguous_kv(wl))
    np.testing.assert_allclose(run.out, ref, rtol=0, atol=1e-12)


def test_fork_workload_matches_sdpa():
    wl = W.best_of_n("bo3", 21, num_groups=2, n_forks=3, prompt_len=40,
                     shared_extra_max=7, private_max=20, num_heads=8,
                     num_kv_heads=2, head_dim=64)
    run = oracle.run(wl)
    ref = sdpa_reference(wl, W.contiguous_kv(wl))
    np.testing.assert_allclose(run.out, ref, rtol=0, atol=1e-12)


def test_invariant_under_block_permutation():
    wl = W.simple("perm", 31, [100, 37, 250], [1, 3, 2], 8, 2, 64, "bf16", pool_factor=2.0)
    a = oracle.run(wl).out
    for seed in (1, 2, 3):
        b = oracle.run(W.with_free_order(wl, seed)).out
        assert np.array_equal(a, b)          # bit-identical: the gather hides placement


def test_identical_keys_give_mean_of_values():
    wl = W.simple("samekey", 41, [23, 64, 9], [1, 1, 1], 4, 2, 64, "f16")
    for op in wl.phases[0] + wl.step:
        if isinstance(op, W.Append):
            op.k[:] = wl.step[0].k[0:1]       # one key row everywhere
    run = oracle.run(wl)
    for s, (K, V) in enumerate(W.contiguous_kv(wl)):
        mean = V.double().mean(0).numpy()                      # [Hkv, d]
        G = wl.num_heads // wl.num_kv_heads
        for h in range(wl.num_heads):
            np.testing.assert_allclose(run.out[s, h], mean[h // G], rtol=0, atol=1e-12)


def test_dominant_logit_selects_its_value_row():
    wl = W.simple("dominant", 42, [50, 80], [1, 1], 2, 2, 64, "f16")
    targets = []
    for s in range(2):
        t_star = 17 + s * 11
        (pre,) = [op for op in wl.phases[0] if isinstance(op, W.Append) and op.seq == s]
        qs = wl.q[s]                                           # [H=2, d]
        pre.k[t_star] = (qs * 64).to(pre.k.dtype)              # logit ~ scale*64*|q|^2 >> others
        targets.append(t_star)
    run = oracle.run(wl)
    for s, (K, V) in enumerate(W.contiguous_kv(wl)):
        for h in range(2):
            logits = wl.scale * (K[:, h].double() @ wl.q[s, h].double())
            srt = torch.sort(logits, descending=True).values
            assert float(srt[0] - srt[1]) > 60.0
            np.testing.assert_allclose(run.out[s, h], V[targets[s], h].double().numpy(),
                                       rtol=0, atol=1e-12)


def test_single_token_context_returns_its_value():
    wl = W.simple("L1", 43, [1, 1], [1, 1], 4, 1, 64, "bf16")
    run = oracle.run(wl)
    for s in range(2):
        v0 = wl.step[s].v[0, 0].double().numpy()
        for h in range(4):
            assert np.array_equal(run.out[s, h], v0)


def test_split_partitions_merge_to_unsplit():
    # ragged lengths across partitions of 128; verify runs that straddle a boundary,
    # so some (row, partition) pairs see no key at all (m=-inf, l=0)
    wl = W.simple("split", 51, [513, 130, 384, 129, 700], [5, 1, 3, 2, 4], 8, 2, 64, "bf16",
                  key_row_boost=8.0, boost_fraction=0.05)
    run = oracle.run(wl)
    P = 128
    nparts = (max(wl.context_lens) + P - 1) // P
    parts = [oracle.attend(run.q64, run.cache, run.block_tables, run.context_lens,
                           wl.query_start_loc, wl.num_heads, wl.scale, p * P, (p + 1) * P)
             for p in range(nparts)]
    o = np.stack([p[0] for p in parts])
    m = np.stack([p[1] for p in parts])
    l = np.stack([p[2] for p in parts])
    assert np.isneginf(m).any() and (l == 0).any()          # an empty partition occurs
    merged = oracle.lse_merge(o, m, l)
    np.testing.assert_allclose(merged, run.out, rtol=0, atol=1e-12)
    # with one partition the merge is the identity
    np.testing.assert_allclose(oracle.lse_merge(run.out[None], run.extra["m"][None],
                                                run.extra["l"][None]), run.out,
                               rtol=0, atol=1e-15)


# ---- planted mistakes: each must be caught by a pin ------------------------

def test_pins_catch_wrong_gqa_head_map():
    wl = small_cases()[1]
    run = oracle.run(wl)
    wrong = sdpa_reference(wl, W.contiguous_kv(wl), gqa="modulo")
    assert np.abs(run.out - wrong).max() > 1e-2


def test_pins_catch_off_by_one_causal_bound():
    wl = small_cases()[2]
    run = oracle.run(wl)
    wrong = sdpa_reference(wl, W.contiguous_kv(wl), causal_shift=-1)
    assert np.abs(run.out - wrong).max() > 1e-2


def test_pins_catch_lost_scale():
    wl = small_cases()[0]
    run = oracle.run(wl)
    wrong = sdpa_reference(wl, W.contiguous_kv(wl), scale=1.0)
    assert np.abs(run.out - wrong).max() > 1e-2


def test_pins_catch_wrong_gather():
    wl = small_cases()[1]
    run = oracle.run(wl)
    bt = run.block_tables.copy()
    s = int(np.argmax((bt >= 0).sum(1)))
    bt[s, 0] = bt[s, 1]               # logical block 0 read from block 1's storage
    o, _, _ = oracle.attend(run.q64, run.cache, bt, run.context_lens, wl.query_start_loc,
                            wl.num_heads, wl.scale)
    ref = sdpa_reference(wl, W.contiguous_kv(wl))
    assert np.abs(o - ref).max() > 1e-6


def test_int8_cache_attends_over_dequantised_values():
    """INT8: the oracle attends over (x_q - zp) * scale (fp32). Gather the codes
    with plain numpy indexing, dequantise in numpy fp32, and compare with SDPA."""
    wl = W.simple("int8", 61, [40, 17, 90], [1, 3, 2], 8, 1, 64, "int8")
    run = oracle.run(wl)
    c = run.cache
    kv_list = []
    for s, L in enumerate(run.context_lens):
        t = np.arange(L)
        blk = run.block_tables[s, t // 16]
        off = t % 16
        ks = c.k[blk, :, off, :].astype(np.int32) - c.k_zp[blk, :, off][..., None]
        vs = c.v[blk, :, off, :].astype(np.int32) - c.v_zp[blk, :, off][..., None]
        K = ks.astype(np.float32) * c.k_scale[blk, :, off][..., None]
        V = vs.astype(np.float32) * c.v_scale[blk, :, off][..., None]
        kv_list.append((torch.from_numpy(K), torch.from_numpy(V)))
    ref = sdpa_reference(wl, kv_list)
    np.testing.assert_allclose(run.out, ref, rtol=0, atol=1e-12)
    # and the dequantised keys are close to the originals (round-trip bound)
    for (K, V), (K0, V0) in zip(kv_list, W.contiguous_kv(wl)):
        err = (K.double() - K0.double()).abs().max().item()
        assert err < 0.02


@pytest.mark.parametrize("step_q_max", [1, 4])
def test_shared_prefix_cascade_equals_full_attention(step_q_max):
    """Read-once decode for forks: attending a group's shared prefix [0, P)
    with all of the group's rows, then each fork's own tokens [P, L), and
    merging the two by log-sum-exp gives the unsplit attention (the prefix
    precedes every query, so the causal bound never cuts it)."""
    wl = W.best_of_n("bo_cascade", 61, num_groups=3, n_forks=4, prompt_len=70,
                     shared_extra_max=9, private_max=30, num_heads=8, num_kv_heads=2,
                     head_dim=64, step_q_max=step_q_max)
    run = oracle.run(wl)
    seqs = [run.names[s] for s in wl.decode_seqs]
    gs, pl = run.pool.prefix_groups(seqs, wl.q_lens)
    assert len(pl) == 3 and min(pl) >= 64           # every group shares its full prompt blocks
    qsl = wl.query_start_loc
    for g in range(len(pl)):
        a, b = gs[g], gs[g + 1]
        rows = slice(int(qsl[a]), int(qsl[b]))
        sub_qsl = qsl[a:b + 1] - qsl[a]
        args = (run.q64[rows], run.cache, run.block_tables[a:b], run.context_lens[a:b],
                sub_qsl, wl.num_heads, wl.scale)
        pre = oracle.attend(*args, 0, pl[g])
        suf = oracle.attend(*args, pl[g])
        merged = oracle.lse_merge(np.stack([pre[0], suf[0]]), np.stack([pre[1], suf[1]]),
                                  np.stack([pre[2], suf[2]]))
        np.testing.assert_allclose(merged, run.out[rows], rtol=0, atol=1e-12)


def test_fp8_cache_attends_over_dequantised_values():
    """FP8: the oracle attends over E4M3(code) * scale_h (fp32), per-head
    scales calibrated to the data. Gather the codes with numpy indexing,
    decode them with torch's float8_e4m3fn, scale in fp32, compare with SDPA."""
    wl = W.simple("fp8", 62, [40, 17, 90], [1, 3, 2], 8, 2, 64, "fp8")
    run = oracle.run(wl)
    c = run.cache
    ks, vs = wl.head_scales
    kv_list = []
    for s, L in enumerate(run.context_lens):
        t = np.arange(L)
        blk = run.block_tables[s, t // 16]
        off = t % 16
        dk = torch.from_numpy(np.ascontiguousarray(c.k[blk, :, off, :])).view(
            torch.float8_e4m3fn).float().numpy()
        dv = torch.from_numpy(np.ascontiguousarray(c.v[blk, :, off, :])).view(
            torch.float8_e4m3fn).float().numpy()
        K = dk * ks[None, :, None]
        V = dv * vs[None, :, None]
        kv_list.append((torch.from_numpy(K), torch.from_numpy(V)))
    ref = sdpa_reference(wl, kv_list)
    np.testing.assert_allclose(run.out, ref, rtol=0, atol=1e-12)
    # round trip: within half an E4M3 step (relative 2^-4) of the originals
    for (K, V), (K0, V0) in zip(kv_list, W.contiguous_kv(wl)):
        for a, b, sc in ((K, K0, ks), (V, V0, vs)):
            err = (a.double() - b.double()).abs()
            bound = b.double().abs() * 2.0 ** -4 + torch.from_numpy(sc).double()[None, :, None] \
                * 2.0 ** -10
            assert (err <= bound).all()
