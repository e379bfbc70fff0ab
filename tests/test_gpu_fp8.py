"""FP8 (E4M3) KV cache with per-head scales, CUDA path vs the CPU oracle:
appended codes bit-identical (the whole pool, canary blocks included),
attention within max abs error 2e-3 of the oracle's attention over the
dequantised cache (fp16 tensor-core products, fp32 accumulate)."""
import numpy as np
import pytest
import torch

import oracle
import workloads as W
import paged_kv_cache_154_gb300 as pa
from gpu_harness import check_cache_bits, check_out, run_both

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    from paged_kv_cache_154_gb300 import build
    build.build()
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"


FP8_SMALL = [
    # name, lens, q_lens, H, Hkv, d, q dtype
    ("fp8_gqa4_d128", [1, 15, 16, 17, 100, 513, 1500], [1] * 7, 32, 8, 128, torch.bfloat16),
    ("fp8_mha_d64_f16q", [33, 700, 64, 129], [1, 1, 1, 1], 4, 4, 64, torch.float16),
    ("fp8_gqa8_verify", [40, 5, 600, 1030, 77], [5, 5, 2, 4, 1], 16, 2, 128, torch.bfloat16),
    ("fp8_mqa_chunks", [300, 1000, 77, 2600], [5, 1, 3, 4], 32, 1, 128, torch.bfloat16),
]


@pytest.mark.parametrize("case", FP8_SMALL, ids=lambda c: c[0])
def test_fp8_small_shapes(case):
    name, lens, qlens, H, Hkv, d, qdt = case
    wl = W.simple(name, 500 + len(lens), lens, qlens, H, Hkv, d, "fp8", q_dtype=qdt)
    ref, cache, si, out = run_both(wl)
    check_cache_bits(ref, cache)
    check_out(ref, out, "fp8")


def test_fp8_llama3_8b_config():
    wl = W.llama3_8b_fp8()
    ref, cache, si, out = run_both(wl)
    check_cache_bits(ref, cache)
    check_out(ref, out, "fp8")


def test_fp8_output_in_q_dtype():
    wl = W.simple("fp8_bf16out", 520, [100, 513, 31], [1, 2, 1], 16, 4, 128, "fp8",
                  q_dtype=torch.bfloat16)
    ref, cache, si, out = run_both(wl, out_dtype=torch.bfloat16)
    check_out(ref, out, "fp8", torch.bfloat16)


def test_fp8_copy_on_write_forks():
    wl = W.best_of_n("fp8_bo3", 521, num_groups=2, n_forks=3, prompt_len=150,
                     shared_extra_max=9, private_max=40, num_heads=16, num_kv_heads=4,
                     head_dim=128, kv_dtype="fp8")
    ref, cache, si, out = run_both(wl)
    check_cache_bits(ref, cache)
    check_out(ref, out, "fp8")


def test_fp8_append_saturates_like_the_oracle():
    """Values far outside the calibrated range saturate to +-448 codes on both
    sides (bit-identical caches), and values in the subnormal range round the
    same way."""
    wl = W.simple("fp8_sat", 522, [40, 20], [1, 1], 8, 2, 64, "fp8", q_dtype=torch.float16)
    for op in wl.phases[0]:
        if isinstance(op, W.Append):
            op.k[::3] = op.k[::3] * 64          # past 448 * scale: saturates
            op.v[1::4] = op.v[1::4] * 2.0 ** -12  # into the E4M3 subnormals
    ref, cache, si, out = run_both(wl)
    check_cache_bits(ref, cache)
    check_out(ref, out, "fp8")
    codes = cache.k.view(torch.uint8).cpu().numpy()
    assert ((codes & 0x7F) == 0x7E).any()       # some codes are the saturated +-448


def test_fp8_graph_replay_matches_eager():
    wl = W.simple("fp8_graph", 523, [200, 50, 1000], [1, 1, 1], 32, 8, 128, "fp8",
                  q_dtype=torch.bfloat16)
    ref, cache, si, out = run_both(wl)
    eager = out.clone()
    g = cache.capture(cache.attend_step, si, wl.scale)
    si.out.zero_()
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(si.out, eager)
