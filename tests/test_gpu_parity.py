"""CUDA path vs the CPU oracle on the same seeded inputs (needs a GB300).

Append and block copies must match bit for bit (the whole pool, canary
blocks included); attention within max abs error 2e-3 for 16-bit caches
(fp32 accumulate, fp32 output)."""
import numpy as np
import pytest
import torch

import oracle
import workloads as W
import paged_kv_cache_154_gb300 as pa
from gpu_harness import check_cache_bits, check_out, run_both, THREADS

pytestmark = pytest.mark.gpu
ARRIVAL_BYTES = pa.ARRIVAL_BYTES   # the counters at the start of every workspace


@pytest.fixture(scope="module", autouse=True)
def built():
    from paged_kv_cache_154_gb300 import build
    build.build()
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"


SMALL = [
    # name, lens, q_lens, H, Hkv, d, dtype, partition
    ("gqa4_bf16_d128", [1, 15, 16, 17, 100, 513, 1000, 1500], [1] * 8, 32, 8, 128, "bf16", 0),
    ("gqa4_bf16_p128", [1, 15, 16, 17, 100, 513, 1000, 1500], [1] * 8, 32, 8, 128, "bf16", 128),
    ("gqa8_bf16", [300, 777, 64, 2049], [1] * 4, 64, 8, 128, "bf16", 256),
    ("mha_f16_d64", [5, 33, 700], [1] * 3, 4, 4, 64, "f16", 0),
    ("mqa16_f16_d64", [90, 1024, 31], [1] * 3, 16, 1, 64, "f16", 512),
    ("verify_gqa4", [40, 5, 600, 1030, 77], [5, 5, 2, 4, 1], 16, 4, 128, "bf16", 512),
    ("verify_gqa8_2tiles", [513, 1026, 96, 2000], [4, 3, 2, 1], 32, 4, 128, "bf16", 512),
    ("verify_straddles_partition", [513, 514, 517], [5, 5, 5], 8, 2, 64, "bf16", 512),
    ("max_partition", [4096, 4097, 9000], [1, 1, 1], 16, 4, 128, "bf16", 4096),
]


@pytest.mark.parametrize("case", SMALL, ids=lambda c: c[0])
def test_small_shapes(case):
    name, lens, qlens, H, Hkv, d, dt, part = case
    wl = W.simple(name, 100 + len(name), lens, qlens, H, Hkv, d, dt)
    ref, cache, si, out = run_both(wl, partition_size=part)
    check_cache_bits(ref, cache)
    check_out(ref, out, dt)


def test_comparison_detects_a_dropped_block():
    """The comparison sees a kernel that skips one block: the CUDA side gets a
    valid but different input -- one sequence's length 16 tokens short, its
    block table unchanged -- and its output must fail against the oracle's
    full-length result (and stay equal to it elsewhere)."""
    wl = W.simple("dropped_block", 99, [300, 1000, 700], [1, 1, 1], 32, 8, 128, "bf16")
    ref, cache, si, out = run_both(wl)
    check_out(ref, out, "bf16")
    short = si.context_lens.clone()
    short[1] -= 16
    out2 = torch.empty_like(si.out)
    pa.decode(out2, si.q, cache.k, cache.v, si.block_tables, short, si.max_context_len, wl.scale,
              None, 1, cache.num_blocks, workspace=si.workspace)
    torch.cuda.synchronize()
    assert (code := pa.device_error()) == 0, hex(code)
    with pytest.raises(AssertionError):
        check_out(ref, out2, "bf16")
    # sequences 0 and 2 (one query token each) are untouched
    err_other = np.abs(out2.double().cpu().numpy()[[0, 2]] - ref.out[[0, 2]]).max()
    assert err_other <= 1e-4, err_other


def test_tiny_config():
    wl = W.tiny()
    ref, cache, si, out = run_both(wl)
    check_cache_bits(ref, cache)
    check_out(ref, out, "f16")
    # and forced through the split-KV path (partitions of one block)
    _, _, _, out2 = run_both(wl, partition_size=16, oracle_run=ref)
    check_out(ref, out2, "f16")


@pytest.mark.parametrize("out_dtype", [torch.bfloat16])
def test_output_in_q_dtype(out_dtype):
    wl = W.simple("outbf16", 7, [100, 700, 1300], [1, 2, 1], 32, 8, 128, "bf16")
    ref, cache, si, out = run_both(wl, out_dtype=out_dtype)
    check_out(ref, out, "bf16", out_dtype)


def test_partials_match_oracle_partitions():
    """Split-KV partition outputs (o normalised, m in base-2 units, l) in the
    workspace agree with the oracle over the same key ranges."""
    P = 256
    wl = W.simple("partials", 9, [700, 256, 1025], [1, 3, 2], 16, 4, 128, "bf16",
                  key_row_boost=8.0, boost_fraction=0.02)
    ref, cache, si, out = run_both(wl, partition_size=P)
    check_out(ref, out, "bf16")
    nq, H, D = si.out.shape
    nparts = (si.max_context_len + P - 1) // P
    ws = si.workspace[ARRIVAL_BYTES:]                  # the partitions' layout follows the counters
    rows = nq * H * nparts
    o_bytes = ((rows * D * 4 + 255) // 256) * 256
    m_bytes = ((rows * 4 + 255) // 256) * 256
    o_part = ws[:rows * D * 4].view(torch.float32).view(nq, H, nparts, D).cpu().numpy()
    m_part = ws[o_bytes:o_bytes + rows * 4].view(torch.float32).view(nq, H, nparts).cpu().numpy()
    l_part = ws[o_bytes + m_bytes:o_bytes + m_bytes + rows * 4].view(torch.float32).view(
        nq, H, nparts).cpu().numpy()
    qsl = wl.query_start_loc
    for p in range(nparts):
        o, m, l = oracle.attend(ref.q64, ref.cache, ref.block_tables, ref.context_lens, qsl,
                                wl.num_heads, wl.scale, p * P, (p + 1) * P)
        for s, L in enumerate(wl.context_lens):
            if L <= P or p * P >= L:
                continue                          # single partition / partition not launched
            rs = slice(qsl[s], qsl[s + 1])
            seen = l[rs] > 0
            np.testing.assert_allclose(o_part[rs, :, p][seen], o[rs][seen], rtol=0, atol=2e-3)
            np.testing.assert_allclose(m_part[rs, :, p][seen], m[rs][seen] * np.log2(np.e),
                                       rtol=1e-5, atol=1e-4)
            np.testing.assert_allclose(l_part[rs, :, p][seen], l[rs][seen], rtol=1e-4)
            assert (l_part[rs, :, p][~seen] == 0).all()
            assert np.isneginf(m_part[rs, :, p][~seen]).all()


def test_llama3_8b_config():
    wl = W.llama3_8b()
    ref, cache, si, out = run_both(wl)
    check_cache_bits(ref, cache)
    check_out(ref, out, "bf16")


def test_best_of_5_copy_on_write_config():
    wl = W.llama2_70b_best_of_5()
    ref, cache, si, out = run_both(wl)
    assert si.pairs is not None and si.pairs.shape[0] >= 8       # the step copies shared tails
    check_cache_bits(ref, cache)
    check_out(ref, out, "bf16")
    free, used, shared = cache.pool.stats()
    assert (free, used, shared) == ref.pool.stats()


@pytest.mark.slow
def test_long_context_split_kv_config():
    wl = W.long_context()
    ref, cache, si, out = run_both(wl)
    check_cache_bits(ref, cache)
    check_out(ref, out, "bf16")


def test_bad_block_id_is_reported_not_faulted():
    wl = W.simple("badblk", 5, [40, 70], [1, 1], 8, 2, 64, "bf16")
    ref, cache, si, out = run_both(wl)
    bt = si.block_tables.clone()
    bt[1, 2] = wl.num_blocks + 1000               # outside the pool
    pa.decode(si.out, si.q, cache.k, cache.v, bt, si.context_lens, si.max_context_len,
              wl.scale, num_blocks=cache.num_blocks, workspace=si.workspace)
    assert pa.device_error() & pa.DEVERR_BAD_BLOCK      # reported, no fault
    assert pa.device_error() == 0                  # the word was cleared


def test_validate_mode_rejects_bad_tables(monkeypatch):
    wl = W.simple("validate", 6, [40, 70], [1, 1], 8, 2, 64, "bf16")
    ref, cache, si, out = run_both(wl)
    monkeypatch.setenv("PA_VALIDATE", "1")
    bt = si.block_tables.clone()
    bt[0, 0] = -5
    with pytest.raises(pa.PAError) as e:
        pa.decode(si.out, si.q, cache.k, cache.v, bt, si.context_lens, si.max_context_len,
                  wl.scale, num_blocks=cache.num_blocks, workspace=si.workspace)
    assert e.value.status == 6
    bad = si.slots.clone()
    bad[0] = cache.num_blocks * 16 + 3
    with pytest.raises(pa.PAError) as e:
        pa.append_kv(si.key, si.value, cache.k, cache.v, bad, cache.num_blocks)
    assert e.value.status == 6
    # valid inputs still pass validation
    pa.decode(si.out, si.q, cache.k, cache.v, si.block_tables, si.context_lens,
              si.max_context_len, wl.scale, num_blocks=cache.num_blocks, workspace=si.workspace)
    torch.cuda.synchronize()


def test_empty_inputs_are_no_ops():
    wl = W.simple("empty", 8, [20], [1], 8, 2, 64, "bf16")
    ref, cache, si, out = run_both(wl)
    before = cache.k.clone()
    pa.append_kv(si.key[:0], si.value[:0], cache.k, cache.v, si.slots[:0], cache.num_blocks)
    pa.decode(si.out[:0], si.q[:0], cache.k, cache.v, si.block_tables[:0], si.context_lens[:0],
              si.max_context_len, wl.scale, num_blocks=cache.num_blocks)
    torch.cuda.synchronize()
    assert torch.equal(before, cache.k)


def _written_slots(ws: torch.Tensor, wl, max_q_len: int):
    """Partial slots of the balanced schedule that the last call wrote (the
    workspace past its arrival counters was filled with 0xFF first, so
    unwritten headers read -1). Layout: the counters, prefix
    sums (num_seqs + 1 int32, 256-byte aligned), then slots of a 32-byte
    header {seq, kv head, chunk, first token, end token} and fp32 m[RT],
    l[RT], O[RT][d]; each entry ends with the slot's index."""
    G = wl.num_heads // wl.num_kv_heads
    rt = 16 if G * max_q_len <= 16 else 64          # rows per tile of the 16-bit kernels
    slot_bytes = (32 + 4 * rt * (wl.head_dim + 2) + 15) // 16 * 16
    cum_bytes = (4 * (wl.num_seqs + 1) + 255) // 256 * 256
    raw = ws.cpu().numpy()[ARRIVAL_BYTES + cum_bytes:]
    out = []
    for i in range(raw.size // slot_bytes):
        b = raw[i * slot_bytes:(i + 1) * slot_bytes]
        hdr = b[:32].view(np.int32)
        if hdr[0] < 0:
            continue
        f = b[32:32 + 4 * rt * (2 + wl.head_dim)].view(np.float32)
        m, l, o = f[:rt], f[rt:2 * rt], f[2 * rt:].reshape(rt, wl.head_dim)
        out.append((tuple(int(x) for x in hdr[:5]), rt, m, l, o, i))
    return out


@pytest.mark.parametrize("case", [
    # many short sequences: a share covers several (sequence, kv head) segments
    ("many_short", [1, 2, 3, 17, 31, 33, 5, 64, 100, 7] * 6, [1] * 60, 16, 4, 128),
    # one long sequence and MQA: far more shares than segments, most cut
    ("one_long", [20000], [1], 8, 1, 128),
    # verify runs and GQA 8: 32 rows, one 64-row tile served by two of the CTA's warps
    ("verify_long", [3000, 777, 4100], [4, 1, 3], 32, 4, 128),
    # long GQA sequences: merged inside the decode kernel, the longest cut by
    # far more than eight shares (two-level merge, group partials in slots)
    ("gqa_long_in_kernel", [12000, 5000, 2000], [1, 1, 1], 32, 8, 128),
    # 96 query rows per KV head: two row chunks per (sequence, kv head)
    ("chunked_rows", [2500, 900], [3, 1], 32, 1, 128),
])
def test_balanced_partials_match_oracle(case):
    name, lens, qlens, H, Hkv, d = case
    wl = W.simple(name, 300 + len(lens), lens, qlens, H, Hkv, d, "bf16")
    ref = oracle.run(wl, threads=THREADS, canary_blocks=W.CANARY_BLOCKS,
                     canary_byte=W.CANARY_BYTE)
    from paged_kv_cache_154_gb300.engine import PagedKVCache
    cache = PagedKVCache(wl.num_blocks, wl.num_kv_heads, wl.head_dim, wl.kv_dtype,
                         free_order=wl.free_order)
    names = {}
    for ops in wl.phases:
        cache.run_phase(ops, names)
    si = cache.prepare_step(wl.step, names, wl.q, torch.float32, 0)
    si.workspace.fill_(0xFF)
    si.workspace[:ARRIVAL_BYTES].zero_()
    cache.step(si, wl.scale, 0)
    torch.cuda.synchronize()
    assert (code := pa.device_error()) == 0, hex(code)
    check_out(ref, si.out, "bf16")
    # the decode kernel's merges leave every arrival counter at zero
    assert not si.workspace[:ARRIVAL_BYTES].any()
    slots = _written_slots(si.workspace, wl, si.max_q_len)
    assert slots, "expected at least one cut segment"
    G = wl.num_heads // wl.num_kv_heads
    qsl = wl.query_start_loc
    per_range = {}    # the oracle over one sequence's keys [t0, t1), all heads
    for (s, g, c, t0, t1), rt, m, l, o, _ in slots:
        L = wl.context_lens[s]
        assert 0 <= t0 < t1 <= L and t0 % 16 == 0
        q0, q1 = int(qsl[s]), int(qsl[s + 1])
        if (s, t0, t1) not in per_range:
            per_range[(s, t0, t1)] = oracle.attend(
                ref.q64[q0:q1], ref.cache, ref.block_tables[s:s + 1], ref.context_lens[s:s + 1],
                np.array([0, q1 - q0], np.int32), wl.num_heads, wl.scale, t0, t1)
        om, mm, lm = per_range[(s, t0, t1)]
        r = q1 - q0
        for j in range(min(rt, G * r - c * rt)):
            row = c * rt + j
            qi, h = row // G, g * G + row % G
            if lm[qi, h] == 0:
                assert l[j] == 0 and np.isneginf(m[j])
                continue
            # m is the partial's reference (base 2): the row's largest logit, or,
            # where a kernel moves it lazily, a logit at most 2^8 below it; l and
            # O are relative to it, which is all the log-sum-exp merge uses
            mx = mm[qi, h] * np.log2(np.e)
            assert m[j] <= mx + 1e-4 and mx <= m[j] + 8 + 1e-4, (m[j], mx)
            np.testing.assert_allclose(l[j] * np.exp2(m[j] - mx), lm[qi, h], rtol=1e-4)
            np.testing.assert_allclose(o[j] / l[j], om[qi, h], rtol=0, atol=2e-3)


def _balanced_state(name, lens, qlens, H, Hkv, d, seed):
    from paged_kv_cache_154_gb300.engine import PagedKVCache
    wl = W.simple(name, seed, lens, qlens, H, Hkv, d, "bf16")
    cache = PagedKVCache(wl.num_blocks, wl.num_kv_heads, wl.head_dim, wl.kv_dtype,
                         free_order=wl.free_order)
    names = {}
    for ops in wl.phases:
        cache.run_phase(ops, names)
    si = cache.prepare_step(wl.step, names, wl.q, torch.float32, 0)
    cache.write_step(si)
    return wl, cache, si


def test_one_workspace_serves_calls_of_any_shape():
    """One buffer, zeroed once, serves a run of calls of different shapes:
    the arrival counters sit at its start whatever the shape, and every call
    leaves them at zero, whether the decode kernel merged its own cut
    segments (the two long GQA calls: one- and two-level merges) or the
    reduce kernel did (a small call, the 64-row kernel). The rest of the
    buffer starts as stale bytes."""
    cases = [("ws_gqa_long", [12000, 5000, 2000], [1, 1, 1], 32, 8, 128),
             ("ws_many_short", [1, 2, 3, 17, 31, 33, 5, 64, 100, 7] * 6, [1] * 60, 16, 4, 128),
             ("ws_verify_rows", [3000, 777, 4100], [4, 1, 3], 32, 4, 128),
             ("ws_d64_in_kernel", [9000, 6000, 3000, 2000], [1, 1, 1, 1], 16, 8, 64)]
    states = [_balanced_state(*c, seed=500 + i) for i, c in enumerate(cases)]
    refs = [oracle.run(wl, threads=THREADS) for wl, _, _ in states]
    big = torch.zeros(max(si.workspace.numel() for _, _, si in states), dtype=torch.uint8,
                      device="cuda")
    big[ARRIVAL_BYTES:].fill_(0x5A)
    for _ in range(2):
        for (wl, cache, si), ref in zip(states, refs):
            si.out.fill_(float("nan"))
            pa.decode(si.out, si.q, cache.k, cache.v, si.block_tables, si.context_lens,
                      si.max_context_len, wl.scale, si.query_start_loc, si.max_q_len,
                      cache.num_blocks, workspace=big)
            torch.cuda.synchronize()
            assert (code := pa.device_error()) == 0, hex(code)
            check_out(ref, si.out, "bf16")
            assert not big[:ARRIVAL_BYTES].any()


@pytest.mark.parametrize("fill", [0x40, 0xFF])
def test_nonzero_arrival_counters_are_reported(fill):
    """Counters that were not zeroed are reported in the device error word
    (no fault, no hang), including 0xFF-poisoned ones that an addition wraps
    around; zeroed again, the next call is correct."""
    # long GQA sequences: the decode kernel merges (and counts) itself
    wl, cache, si = _balanced_state("ws_dirty", [12000, 3000, 3000], [1, 1, 1], 32, 8, 128,
                                    seed=510)
    ref = oracle.run(wl, threads=THREADS)
    args = (si.q, cache.k, cache.v, si.block_tables, si.context_lens, si.max_context_len,
            wl.scale, si.query_start_loc, si.max_q_len, cache.num_blocks)
    si.workspace[:ARRIVAL_BYTES].fill_(fill)       # every counter past any segment's total
    pa.decode(si.out, *args, workspace=si.workspace)
    torch.cuda.synchronize()
    assert pa.device_error() & pa.DEVERR_WORKSPACE
    si.workspace[:ARRIVAL_BYTES].zero_()
    si.out.fill_(float("nan"))
    pa.decode(si.out, *args, workspace=si.workspace)
    torch.cuda.synchronize()
    assert (code := pa.device_error()) == 0, hex(code)
    check_out(ref, si.out, "bf16")
    assert not si.workspace[:ARRIVAL_BYTES].any()


def test_int8_tensor_core_writes_stay_inside_workspace_and_output():
    """The INT8 tensor-core kernel's 96-row partial slots: a call sized by the
    workspace query writes nothing past it nor past the output, leaves the
    arrival counters zero, and matches the oracle."""
    from paged_kv_cache_154_gb300.engine import PagedKVCache
    wl = W.simple("int8_tc_ws", 530, [9000, 40, 2500, 600, 1800], [3, 2, 5, 4, 2], 32, 1, 128,
                  "int8")
    cache = PagedKVCache(wl.num_blocks, wl.num_kv_heads, wl.head_dim, wl.kv_dtype,
                         free_order=wl.free_order)
    names = {}
    for ops in wl.phases:
        cache.run_phase(ops, names)
    si = cache.prepare_step(wl.step, names, wl.q, torch.float32, 0)
    cache.write_step(si)
    ref = oracle.run(wl, threads=THREADS)
    need = si.workspace.numel()
    ws = torch.full((need + (1 << 16),), 0xA5, dtype=torch.uint8, device="cuda")
    ws[:ARRIVAL_BYTES].zero_()
    nq = si.out.shape[0]
    out = torch.full((nq + 4,) + tuple(si.out.shape[1:]), float("nan"), device="cuda")
    pa.decode(out[:nq], si.q, cache.k, cache.v, si.block_tables, si.context_lens,
              si.max_context_len, wl.scale, si.query_start_loc, si.max_q_len, cache.num_blocks,
              cache.k_scale, cache.v_scale, cache.k_zp, cache.v_zp, workspace=ws[:need])
    torch.cuda.synchronize()
    assert (code := pa.device_error()) == 0, hex(code)
    check_out(ref, out[:nq], "int8")
    assert bool((ws[need:] == 0xA5).all()), "bytes written past the workspace"
    assert bool(out[nq:].isnan().all()), "rows written past the output"
    assert not ws[:ARRIVAL_BYTES].any()


@pytest.mark.parametrize("case", [
    ("spare_warps_mqa", [20000], [1], 8, 1, 128),        # 1250 workers: 2 spare warps
    ("spare_warps_d64", [1000, 77], [1, 1], 4, 1, 64),   # 2 x 63 = 126 workers, 68 blocks
])
def test_writes_stay_inside_workspace_and_output(case):
    """Calls whose worker count is not a multiple of the CTA's four warps
    (the grid's last CTA has spare warps): nothing is written past the
    workspace the size query asked for, nor past the output, and the output
    matches the oracle."""
    name, lens, qlens, H, Hkv, d = case
    wl, cache, si = _balanced_state(name, lens, qlens, H, Hkv, d, seed=520)
    ref = oracle.run(wl, threads=THREADS)
    need = si.workspace.numel()
    guard = 1 << 16
    ws = torch.full((need + guard,), 0xA5, dtype=torch.uint8, device="cuda")
    ws[:ARRIVAL_BYTES].zero_()
    nq = si.out.shape[0]
    out = torch.full((nq + 4,) + tuple(si.out.shape[1:]), float("nan"), device="cuda")
    pa.decode(out[:nq], si.q, cache.k, cache.v, si.block_tables, si.context_lens,
              si.max_context_len, wl.scale, si.query_start_loc, si.max_q_len, cache.num_blocks,
              workspace=ws[:need])
    torch.cuda.synchronize()
    assert (code := pa.device_error()) == 0, hex(code)
    check_out(ref, out[:nq], "bf16")
    assert bool((ws[need:] == 0xA5).all()), "bytes written past the workspace"
    assert bool(out[nq:].isnan().all()), "rows written past the output"
    assert not ws[:ARRIVAL_BYTES].any()


def test_many_query_rows_per_kv_head_use_row_chunks():
    """MQA with 32 q heads and verify runs of up to 5 tokens: up to 160 query
    rows per KV head, served as row tiles of 64 (three chunks re-reading the
    same KV), checked against the oracle."""
    wl = W.simple("mqa_rows160", 71, [300, 1000, 77, 2600, 16, 5], [5, 1, 3, 4, 2, 5], 32, 1,
                  128, "bf16")
    ref, cache, si, out = run_both(wl)
    check_cache_bits(ref, cache)
    check_out(ref, out, "bf16")


INT8_SMALL = [
    # name, lens, q_lens, H, Hkv, d, q dtype
    ("int8_gqa4", [1, 15, 16, 17, 100, 513, 1500], [1] * 7, 32, 8, 128, torch.bfloat16),
    ("int8_mqa_verify", [5, 40, 300, 1025, 2000, 77], [5, 2, 1, 4, 3, 5], 32, 1, 128,
     torch.bfloat16),
    ("int8_d64_f16q", [33, 700, 64, 129], [1, 2, 1, 3], 8, 2, 64, torch.float16),
    ("int8_mha", [200, 31], [1, 1], 4, 4, 128, torch.bfloat16),
    # 64 query rows per KV head on average at d = 128 (the tensor-core
    # kernel, tokens in M): contexts of 1 and 2 tokens, partial tiles, a long
    # sequence cut across many shares, fp16 q
    ("int8_mqa_tc_f16q", [1, 2, 17, 64, 65, 4097, 333, 16], [1, 1, 2, 1, 5, 1, 4, 1], 32, 1,
     128, torch.float16),
    # GQA verify runs, 26 rows on average (the per-warp kernel's row chunks)
    ("int8_gqa8_verify", [900, 45, 3000, 7], [4, 5, 3, 1], 32, 4, 128, torch.bfloat16),
    # the tensor-core kernel: 40 sequences of 64 rows whose blocks are cut
    # into pieces across the CTAs' shares (partial slots and their merge)
    ("int8_tc_rows64_many", [50 + (37 * i * i) % 4900 for i in range(40)], [2] * 40, 32, 1, 128,
     torch.bfloat16),
    # the tensor-core kernel with two KV heads and 16 q heads each: 48 and 80
    # rows (column padding to 64 and 96), causal verify masks, fp16 q
    ("int8_tc_gqa16_verify", [1200, 33, 2600, 700, 129, 3100], [3, 5, 4, 5, 3, 4], 32, 2, 128,
     torch.float16),
]


@pytest.mark.parametrize("case", INT8_SMALL, ids=lambda c: c[0])
def test_int8_small_shapes(case):
    """INT8 KV: codes, scales and zero points bit-identical to the oracle's
    quantiser; attention over the dequantised values within 1e-2."""
    name, lens, qlens, H, Hkv, d, qdt = case
    wl = W.simple(name, 500 + len(name), lens, qlens, H, Hkv, d, "int8", q_dtype=qdt,
                  key_row_boost=4.0, boost_fraction=0.02)
    ref, cache, si, out = run_both(wl)
    check_cache_bits(ref, cache)
    check_out(ref, out, "int8")


@pytest.mark.parametrize("qlens", [[2, 1], [3, 2]], ids=["per_warp", "tensor_core"])
@pytest.mark.parametrize("qdt", [torch.bfloat16, torch.float16], ids=["bf16", "f16"])
def test_int8_output_in_q_dtype(qdt, qlens):
    wl = W.simple("int8_out16", 77, [300, 1000], qlens, 32, 1, 128, "int8", q_dtype=qdt)
    ref, cache, si, out = run_both(wl, out_dtype=qdt)
    check_out(ref, out, "int8", qdt)


def test_mixed_int8_config():
    """256 ragged sequences, MQA 32/1, INT8 KV, 20% with verify runs of 2-5."""
    wl = W.mixed_int8()
    ref, cache, si, out = run_both(wl)
    check_cache_bits(ref, cache)
    check_out(ref, out, "int8")


@pytest.mark.parametrize("heads,qlens", [((16, 2), [1, 3, 1]), ((32, 1), [1, 3, 1]),
                                         ((32, 1), [4, 5, 3])],
                         ids=["gqa8", "mqa32", "mqa32_tensor_core"])
def test_int8_wide_value_range(heads, qlens):
    """K/V rows scaled by 2^-6 .. 2^0 (per token and head) and q rows by
    2^-6 .. 2^6: the running power-of-two V reference must keep the small
    rows, and the per-row power-of-two q scaling must make the fp16
    conversion of q exact. (Outputs stay of order one, the regime the 1e-2
    tolerance is stated for; the fp16 weights carry 2^-11 relative error, below
    the INT8 quantisation step of 1/255 of a row's range.)"""
    wl = W.simple("int8_range", 91, [800, 1200, 50], qlens, heads[0], heads[1], 128, "int8",
                  q_dtype=torch.bfloat16)
    rng = np.random.default_rng(0)
    for op in wl.phases[0] + wl.step:
        if isinstance(op, W.Append):
            f = torch.from_numpy(2.0 ** rng.integers(-6, 1, size=op.k.shape[:2])).float()
            op.k[:] = (op.k.float() * f[..., None]).to(op.k.dtype)
            op.v[:] = (op.v.float() * f[..., None]).to(op.v.dtype)
    fq = torch.from_numpy(2.0 ** rng.integers(-6, 7, size=wl.q.shape[:2])).float()
    wl.q[:] = (wl.q.float() * fq[..., None]).to(wl.q.dtype)
    ref, cache, si, out = run_both(wl)
    check_cache_bits(ref, cache)
    check_out(ref, out, "int8")


def test_graph_replay_matches_eager():
    """A step captured in CUDA graphs (writes; attention, with programmatic
    dependent launches) replays to the same bits as the eager calls."""
    wl = W.simple("graph", 17, [700, 2300, 90, 1500], [1, 3, 1, 2], 32, 8, 128, "bf16")
    ref, cache, si, out = run_both(wl)
    eager = out.clone()
    g_write = cache.capture(cache.write_step, si)
    g_attend = cache.capture(cache.attend_step, si, wl.scale, 0)
    si.out.zero_()
    for _ in range(3):
        g_write.replay()
        g_attend.replay()
    torch.cuda.synchronize()
    assert (code := pa.device_error()) == 0, hex(code)
    assert torch.equal(si.out, eager)
    check_cache_bits(ref, cache)


PREFILL = [
    # name, lens (post-append), q_lens, H, Hkv, d, dtype: chunked prefill over cached context
    ("prefill_fresh_gqa4", [64, 200, 128], [64, 200, 128], 32, 8, 128, "bf16"),
    ("prefill_over_context", [164, 900, 1000], [64, 200, 128], 32, 8, 128, "bf16"),
    ("prefill_mha_d64_f16", [300, 90], [150, 90], 8, 8, 64, "f16"),
    ("prefill_mqa", [400, 333], [96, 33], 32, 1, 128, "bf16"),
    # the tensor-core kernel over an fp16 cache; task rows not a multiple of
    # 128 (a half-empty second Q tile), a context ending mid-block
    ("prefill_tc_f16_ragged", [517, 70, 1234], [77, 70, 300], 16, 4, 128, "f16"),
]


@pytest.mark.parametrize("case", PREFILL, ids=lambda c: c[0])
def test_paged_prefill_matches_oracle(case):
    """Long query runs (prefill chunks): causal attention over the paged cache,
    row chunks skip the blocks none of their queries can see."""
    name, lens, qlens, H, Hkv, d, dt = case
    wl = W.simple(name, 600 + len(lens), lens, qlens, H, Hkv, d, dt)
    ref, cache, si, out = run_both(wl)
    check_cache_bits(ref, cache)
    check_out(ref, out, dt)


def test_paged_prefill_peaked_softmax():
    """2% of the key rows scaled by 8: peaked softmaxes whose running max moves
    by more than 2^8 mid-stream (the tensor-core kernel rescales O in TMEM)."""
    wl = W.simple("prefill_peaked", 621, [1500, 640], [320, 256], 32, 8, 128, "bf16",
                  key_row_boost=8.0, boost_fraction=0.02)
    ref, cache, si, out = run_both(wl)
    check_out(ref, out, "bf16")


@pytest.mark.parametrize("dt", ["bf16", "f16"])
def test_paged_prefill_output_in_cache_dtype(dt):
    """The tensor-core prefill kernel writing 16-bit outputs."""
    qdt = torch.bfloat16 if dt == "bf16" else torch.float16
    wl = W.simple("prefill_out16_" + dt, 620, [700, 300], [256, 100], 32, 8, 128, dt)
    ref, cache, si, out = run_both(wl, out_dtype=qdt)
    check_out(ref, out, dt, qdt)


@pytest.mark.parametrize("kv", ["int8", "fp8"])
def test_paged_prefill_quantised_caches(kv):
    wl = W.simple("prefill_" + kv, 610, [300, 700], [120, 64], 32, 8, 128, kv,
                  q_dtype=torch.bfloat16)
    ref, cache, si, out = run_both(wl)
    check_cache_bits(ref, cache)
    check_out(ref, out, kv)


@pytest.mark.slow
def test_paged_prefill_config():
    wl = W.paged_prefill()
    ref, cache, si, out = run_both(wl)
    check_out(ref, out, "bf16")
